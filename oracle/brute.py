"""Pure-Python brute force of paged decode attention (tiny inputs only).

Test infrastructure only.  Written with scalar loops and math.fsum, without
numpy arithmetic, as an independent check of ``paged_decode_attention``:
token t of sequence s lives at row t % bs of block block_table[s][t // bs]
("LLM 서빙과 KV Cache, VLLM", section "PagedAttention"); query head h reads kv
group h // (n_h / n_kv) ("KV Cache는 왜 LLM 서빙의 핵심인가", section "메모리
공식과 GQA의 동기"); the output is softmax(scale q.K^T) V ("KV Cache: O(T²)를
O(T)로", decode-step listing).  With a limited attention window of W tokens only
the last W tokens of the context take part ("KV 캐시 시스템 (KV Cache System)",
section "제한된 어텐션 윈도우 크기 (Limited Attention Window Size)").
"""
import math


def attention_loops(q, k_pool, v_pool, block_tables, context_lens, scale, block_size, window=0):
    """q: nested lists / arrays [B][n_h][d]; returns nested lists [B][n_h][d] of floats."""
    B, n_h, d = len(q), len(q[0]), len(q[0][0])
    n_kv = len(k_pool[0])
    G = n_h // n_kv
    out = []
    for s in range(B):
        L = int(context_lens[s])
        first = L - window if 0 < window < L else 0
        rows = []
        for h in range(n_h):
            if L == 0:
                rows.append([0.0] * d)
                continue
            g = h // G
            logits = []
            for t in range(first, L):
                blk = int(block_tables[s][t // block_size])
                krow = k_pool[blk][g][t % block_size]
                logits.append(scale * math.fsum(float(q[s][h][i]) * float(krow[i]) for i in range(d)))
            mx = max(logits)
            e = [math.exp(x - mx) for x in logits]
            z = math.fsum(e)
            o = []
            for j in range(d):
                acc = []
                for i, t in enumerate(range(first, L)):
                    blk = int(block_tables[s][t // block_size])
                    acc.append(e[i] * float(v_pool[blk][g][t % block_size][j]))
                o.append(math.fsum(acc) / z)
            rows.append(o)
        out.append(rows)
    return out
