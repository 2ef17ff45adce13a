"""KV block manager with cross-request reuse, priority-LRU eviction and host offload,
restated plainly.  Test infrastructure only (see the package header).

Source: "KV 캐시 시스템 (KV Cache System)":

* section "요청 간 재사용 (Reuse Across Requests)": a block stays reusable until it is
  evicted from the search tree; eviction happens when a new (free) block is needed; the
  policy is priority-based LRU with every block carrying a priority from 0 to 100, 100
  the most important.
* section "보존 정책 (Retention Policy)": priorities come from the request's retention
  config, a list of token ranges each with a priority (e.g. tokens 10 to 61 get
  priority X); lower-priority blocks are freed before higher-priority ones.
* section "호스트 메모리로의 오프로딩 (Enable Offloading to Host Memory)": before a block
  is evicted from GPU memory it may be offloaded to host memory, where it stays
  reusable until evicted from there; reusing it copies it back to the GPU first; blocks
  below secondary_offload_min_priority (default 35) are not offloaded but evicted
  directly.
* section "제한된 어텐션 윈도우 크기 (Limited Attention Window Size)": blocks that leave
  a layer's attention window are freed into the search tree, reusable.
* "LLM 서빙과 KV Cache, VLLM", section "PagedAttention": fixed-size blocks anywhere in a
  shared pool, a block table per sequence; slot = block * block_size + row.

Readings where the page is silent (each is also a line of the design notes):

* Search tree: a node is one full block of tokens under its parent node (the root for a
  sequence's first block); its key is the parent plus the block's token ids.  Only full
  blocks enter the tree; a sequence's last, partial block is private.
* Matching: a new request walks the tree over its full prompt blocks and reuses the
  longest matching chain, but always leaves at least one prompt token to compute (at
  most floor((n - 1) / bs) blocks are reused).
* Registration: a block is registered when its last row is allocated (prompt blocks at
  add time, decode blocks when their last token is appended).  If an identical node
  already exists the block stays private, and so do the sequence's later blocks.
* Priority of a block: the highest priority among the request's ranges that overlap
  the block's token positions, else the default priority (35, the offload threshold's
  default, so blocks without a range are offloadable).  A reused node takes the
  priority of the request that reuses it.
* LRU time: a logical clock that advances once per call; a block's time is that of the
  last call that allocated, reused or released it.  Victim = the cached (unreferenced)
  GPU block with the smallest (priority, time, -depth, block id), depth counting the
  node's ancestors, so a request's chain is evicted from its end; host victim likewise
  by (priority, time, -depth, host slot).
* Evicting a cached GPU block: if its priority is at least the offload threshold and a
  host slot is free (or can be freed by evicting a host block), it is offloaded and stays
  in the tree on the host; otherwise it is dropped.  Dropping a node drops its whole
  subtree (a dropped prefix can never be matched again); a block of the subtree still
  held by a request (possible once that request slid its window past the node) leaves
  the tree but stays with the request.
* Free blocks are taken lowest id first.
* Copies: OFFLOAD (gpu block -> host slot) and ONLOAD (host slot -> gpu block) are
  recorded in order and must be applied in that order before the pools are used.
"""
from __future__ import annotations

OFFLOAD, ONLOAD = 0, 1
ROOT = 0


class OutOfBlocks(Exception):
    pass


class BlockManager:
    def __init__(self, num_blocks, block_size, host_blocks=0, offload_min_priority=35, default_priority=35):
        self.N, self.bs, self.H = num_blocks, block_size, host_blocks
        self.offload_min = offload_min_priority
        self.default_priority = default_priority
        self.gpu_ref = [0] * num_blocks
        self.gpu_node = [None] * num_blocks          # node id registered on this block
        self.host_node = [None] * host_blocks
        self.nodes = {}                              # id -> dict(parent, key, children, loc, prio, time)
        self.index = {}                              # (parent id, token tuple) -> node id
        self.next_node = 1
        self.seqs = {}
        self.clock = 0
        self.copies = []
        self.stats = dict(reused_tokens=0, evictions=0, offloads=0, onloads=0, drops=0)

    # ---- helpers --------------------------------------------------------------------------
    def _priority(self, ranges, i):
        lo, hi = i * self.bs, (i + 1) * self.bs
        best = None
        for start, end, prio in ranges:
            e = hi if end < 0 else end
            if start < hi and e > lo:
                best = prio if best is None else max(best, prio)
        return self.default_priority if best is None else best

    def _gpu_state(self, b):
        if self.gpu_ref[b] > 0:
            return "active"
        return "cached" if self.gpu_node[b] is not None else "free"

    def _subtree(self, nid):
        out, stack = [], [nid]
        while stack:
            x = stack.pop()
            out.append(x)
            stack.extend(sorted(self.nodes[x]["children"]))
        return out

    def _drop(self, nid):
        """Remove a node and its subtree from the tree.  Unreferenced GPU blocks and host
        slots of those nodes become free; a block still referenced (a sequence that slid
        its window past the node's ancestors holds it) stays with its sequence, private."""
        for x in self._subtree(nid):
            n = self.nodes.pop(x)
            kind, where = n["loc"]
            if kind == "gpu":
                self.gpu_node[where] = None
            else:
                self.host_node[where] = None
            del self.index[(n["parent"], n["key"])]
            if n["parent"] in self.nodes:
                self.nodes[n["parent"]]["children"].discard(x)
            self.stats["drops"] += 1

    def _host_slot(self):
        """A free host slot, evicting (dropping) a host block if needed; None if impossible."""
        for h in range(self.H):
            if self.host_node[h] is None:
                return h
        cands = [(self.nodes[self.host_node[h]]["prio"], self.nodes[self.host_node[h]]["time"],
                  -self.nodes[self.host_node[h]]["depth"], h) for h in range(self.H) if self.host_node[h] is not None]
        if not cands:
            return None
        h = min(cands)[3]
        self._drop(self.host_node[h])
        return h

    def _evict_one(self):
        cands = [(self.nodes[self.gpu_node[b]]["prio"], self.nodes[self.gpu_node[b]]["time"],
                  -self.nodes[self.gpu_node[b]]["depth"], b) for b in range(self.N) if self._gpu_state(b) == "cached"]
        if not cands:
            raise OutOfBlocks()
        prio, _, _, b = min(cands)
        nid = self.gpu_node[b]
        self.stats["evictions"] += 1
        if prio >= self.offload_min and self.H > 0:
            h = self._host_slot()
            if h is not None and self.gpu_node[b] == nid:      # the host eviction may have dropped it
                self.copies.append((OFFLOAD, b, h))
                self.nodes[nid]["loc"] = ("host", h)
                self.host_node[h] = nid
                self.gpu_node[b] = None
                self.stats["offloads"] += 1
                return
        if self.gpu_node[b] == nid:
            self._drop(nid)

    def _alloc(self):
        while True:
            for b in range(self.N):
                if self._gpu_state(b) == "free":
                    return b
            self._evict_one()

    def _register(self, seq, i, b):
        """Register full block i of seq (on gpu block b) under the sequence's chain."""
        parent = seq["chain"]
        if parent is None or (parent != ROOT and parent not in self.nodes):
            seq["chain"] = None                     # the chain's last node was dropped
            return
        key = tuple(seq["tokens"][i * self.bs:(i + 1) * self.bs])
        if (parent, key) in self.index:
            seq["chain"] = None                     # someone registered the same block first
            return
        nid = self.next_node
        self.next_node += 1
        depth = 1 if parent == ROOT else self.nodes[parent]["depth"] + 1
        self.nodes[nid] = dict(parent=parent, key=key, children=set(), loc=("gpu", b),
                               prio=seq["prios"][i], time=self.clock, depth=depth)
        if parent != ROOT:
            self.nodes[parent]["children"].add(nid)
        self.index[(parent, key)] = nid
        self.gpu_node[b] = nid
        seq["chain"] = nid

    # ---- API ------------------------------------------------------------------------------
    def add_sequence(self, seq_id, tokens, ranges=()):
        """Allocate the blocks of a new request's prompt; returns (block table, reused tokens)."""
        assert seq_id not in self.seqs
        self.clock += 1
        tokens = [int(t) for t in tokens]
        n = len(tokens)
        nb = -(-n // self.bs)
        seq = dict(tokens=tokens, blocks=[], prios=[self._priority(ranges, i) for i in range(nb)],
                   ranges=list(ranges), chain=ROOT, first=0)
        self.seqs[seq_id] = seq
        # longest matching chain of full blocks, leaving at least one token to compute
        matched = []
        parent = ROOT
        for i in range(max(0, (n - 1) // self.bs)):
            nid = self.index.get((parent, tuple(tokens[i * self.bs:(i + 1) * self.bs])))
            if nid is None:
                break
            matched.append(nid)
            parent = nid
        try:
            for i, nid in enumerate(matched):
                node = self.nodes.get(nid)
                if node is None:                    # dropped while making room for an earlier one
                    del matched[i:]
                    break
                kind, where = node["loc"]
                if kind == "host":
                    b = self._alloc()
                    node = self.nodes.get(nid)
                    if node is None or node["loc"] != ("host", where):
                        del matched[i:]                 # making room dropped it
                        break
                    self.copies.append((ONLOAD, where, b))
                    self.host_node[where] = None
                    node["loc"] = ("gpu", b)
                    self.gpu_node[b] = nid
                    self.stats["onloads"] += 1
                else:
                    b = where
                self.gpu_ref[b] += 1
                node["prio"] = seq["prios"][i]
                node["time"] = self.clock
                seq["blocks"].append(b)
                seq["chain"] = nid
            reused = len(seq["blocks"])
            for i in range(reused, nb):
                b = self._alloc()
                self.gpu_ref[b] = 1
                seq["blocks"].append(b)
        except OutOfBlocks:
            self._release(seq_id)                   # nothing new was registered
            raise
        # the prompt's new full blocks enter the tree once all of them have a block
        for i in range(reused, nb):
            if (i + 1) * self.bs <= n:
                self._register(seq, i, seq["blocks"][i])
        self.stats["reused_tokens"] += reused * self.bs
        return list(seq["blocks"]), reused * self.bs

    def append_token(self, seq_id, token):
        """Slot of one new token of a running sequence (a new block when the last is full)."""
        self.clock += 1
        seq = self.seqs[seq_id]
        t = len(seq["tokens"])
        i = t // self.bs
        if t % self.bs == 0:                        # a new block (on failure nothing changes)
            b = self._alloc()
            self.gpu_ref[b] = 1
            seq["blocks"].append(b)
            seq["prios"].append(self._priority(seq["ranges"], i))
        seq["tokens"].append(int(token))
        b = seq["blocks"][i]
        if t % self.bs == self.bs - 1:
            self._register(seq, i, b)
        return b * self.bs + t % self.bs

    def _release_block(self, b):
        self.gpu_ref[b] -= 1
        if self.gpu_ref[b] == 0 and self.gpu_node[b] is not None:
            self.nodes[self.gpu_node[b]]["time"] = self.clock

    def _release(self, seq_id):
        seq = self.seqs.pop(seq_id)
        for b in seq["blocks"][seq["first"]:]:
            self._release_block(b)

    def release(self, seq_id):
        """End of a request: its full registered blocks stay cached, the rest are freed."""
        self.clock += 1
        self._release(seq_id)

    def slide_window(self, seq_id, window):
        """Release the blocks that end before the last `window` tokens of the sequence."""
        self.clock += 1
        seq = self.seqs[seq_id]
        n = len(seq["tokens"])
        first = max(0, n - window) // self.bs if window > 0 else 0
        for i in range(seq["first"], first):
            self._release_block(seq["blocks"][i])
        seq["first"] = max(seq["first"], first)
        return seq["first"]

    def table(self, seq_id):
        seq = self.seqs[seq_id]
        return list(seq["blocks"]), len(seq["tokens"])

    def take_copies(self):
        c, self.copies = self.copies, []
        return c

    def counts(self):
        st = [self._gpu_state(b) for b in range(self.N)]
        return dict(free=st.count("free"), active=st.count("active"), cached=st.count("cached"),
                    host=sum(x is not None for x in self.host_node))


def apply_copies(copies, gpu_pool, host_pool):
    """Apply recorded copies in order to numpy pools ([num_blocks][...] / [host_blocks][...])."""
    for kind, src, dst in copies:
        if kind == OFFLOAD:
            host_pool[dst] = gpu_pool[src]
        else:
            gpu_pool[dst] = host_pool[src]
