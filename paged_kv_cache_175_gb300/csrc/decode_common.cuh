// Work partition shared by the paged decode-attention kernels.
//
// The unit of work is one (sequence s, kv head g, logical block i) triple.  All units
// are laid out on one line in (s, g, i) order: sequence s with nb_s = ceil(ctx_s / bs)
// blocks owns positions [n_kv * cum[s], n_kv * cum[s+1]) where cum is the exclusive
// prefix sum of nb; inside it, kv head g owns the segment starting at
// n_kv * cum[s] + g * nb_s.  The line of W = n_kv * cum[B] positions is cut into P
// equal pieces, piece p = [floor(p W / P), floor((p+1) W / P)), one per CTA of a
// persistent grid, so every CTA streams the same number of K/V tiles whatever the
// mix of context lengths.  A segment cut by piece boundaries leaves one partial
// softmax state per piece it touches, stored at part index (segment + piece), which
// is unique because both indices grow along the line; the reduce kernel merges them.
#pragma once

#include "pkv_device.cuh"

namespace pkv {

enum : int { F_FIRST = 1, F_LAST = 2, F_WHOLE = 4, F_VALID = 8 };
// Ring stages of up to two blocks: F_PAIR marks a stage that also holds the next block of
// the same segment; F_END marks the last stage of a piece.
enum : int { F_PAIR = 16, F_END = 32 };
// Lazy softmax offset (base-2 units): the attention kernels raise a head's running offset
// only when a score exceeds it by more than this, so exponentials stay below 2^8 (well
// inside the range of the fp16 / bf16 high + low split of P) and most tiles skip the max
// reduction and the rescale.  Softmax itself does not depend on the offset.
constexpr float kLazyMax = 8.f;

struct DecodeArgs {
  const void* q;                 // bf16 [B][n_h][D]
  const int32_t* bt;             // [B][max_blocks]
  int max_blocks;
  const int32_t* cum;            // workspace: [B+1] exclusive prefix of blocks per sequence
  const int32_t* ctx_eff;        // workspace: [B] context lengths after range checks
  const int4* pieces;            // workspace: [P][2] start cursor of each piece (s, g, blk, nb | ctx)
  int batch, n_h, n_kv, G, num_blocks;
  float scale_log2;              // scale * log2(e): softmax runs in base 2
  void* out;
  int out_f32;
  float* ws_ml;                  // [parts][G][2] (running max in log2 units, running sum)
  float* ws_o;                   // [parts][G][D] unnormalised partial outputs
  int32_t* err;
  int stages;
  // Without a plan kernel (batch <= kInlinePlanSeqs) the kernels read the raw context
  // lengths and clamp them to [0, max_ctx] themselves.
  const int32_t* ctx_raw;
  int max_ctx, block_size, inline_plan;
  int window;                    // attention window in tokens (0: the whole context)
  // INT4 cache (unused by the bf16 kernel): (block, kv head) records and the bf16 K tail
  const uint8_t* cache;
  const __nv_bfloat16* k_tail;
  int P_launch;                  // CTAs of the attention grid (the reduce derives the pieces)
};

struct WorkspaceLayout {
  size_t cum, ctx, pieces, ml, o, total;
};

// Pieces actually used for a line of W positions when P CTAs are launched: at least
// kMinPiece positions per piece, so a small batch is not cut into one-tile parts whose
// merge would cost more than streaming them.
constexpr int kMinPiece = 8;
__host__ __device__ inline int effective_pieces(long long W, int P) {
  const long long q = (W + kMinPiece - 1) / kMinPiece;
  return (int)(q < 1 ? 1 : (q < P ? q : P));
}

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

__host__ inline WorkspaceLayout workspace_layout(int B, int n_kv, int G, int D, int P) {
  WorkspaceLayout w;
  const size_t parts = (size_t)B * n_kv + (size_t)P;
  w.cum = 0;
  w.ctx = align_up(sizeof(int32_t) * (size_t)(B + 1), 16);
  w.pieces = align_up(w.ctx + sizeof(int32_t) * (size_t)B, 32);
  w.ml = align_up(w.pieces + 2 * sizeof(int4) * (size_t)P, 256);
  w.o = align_up(w.ml + sizeof(float) * parts * G * 2, 256);
  w.total = align_up(w.o + sizeof(float) * parts * G * D, 256);
  return w;
}

// Limited attention window: a sequence of ctx tokens attends to its last `window` tokens,
// [ctx - window, ctx), when window > 0; its segment holds only the blocks from the one
// the window starts in, so blocks before the window are never read.
__host__ __device__ __forceinline__ int window_first_block(int ctx, int window, int bs) {
  return (window > 0 && ctx > window) ? (ctx - window) / bs : 0;
}
// Rows of the window's first block that lie before the window.
__host__ __device__ __forceinline__ int window_lead(int ctx, int window, int bs) {
  return (window > 0 && ctx > window) ? (ctx - window) % bs : 0;
}
// Blocks a sequence's segment covers.
__host__ __device__ __forceinline__ int span_blocks(int ctx, int window, int bs) {
  return (ctx + bs - 1) / bs - window_first_block(ctx, window, bs);
}

// Piece that holds line position pos (the largest p with floor(p W / P) <= pos).
__device__ __forceinline__ int piece_of(long long pos, long long W, int P) {
  return (int)(((pos + 1) * (long long)P - 1) / W);
}

// Warp-uniform cursor over the line of positions.
struct Cursor {
  int s, g, blk, nb, ctx;        // blk counts from the segment's first block
  int b0;                        // logical block of the segment's first block (window start)
  long long seg_start;           // line position of block 0 of segment (s, g)
};

// Start cursor of piece p, precomputed by the plan kernel (one 32-byte load).
__device__ __forceinline__ void cursor_from_table(Cursor& c, int p, long long pstart, const DecodeArgs& a) {
  const int4 e0 = a.pieces[2 * p], e1 = a.pieces[2 * p + 1];
  c.s = e0.x;
  c.g = e0.y;
  c.blk = e0.z;
  c.nb = e0.w;
  c.ctx = e1.x;
  c.b0 = window_first_block(c.ctx, a.window, a.block_size);
  c.seg_start = pstart - c.blk;
}

constexpr int kInlinePlanSeqs = 256;

__device__ __forceinline__ int clamp_ctx(int c, int max_ctx) { return c < 0 ? 0 : (c > max_ctx ? max_ctx : c); }

// The part of the line a CTA owns, computed by one whole warp (every lane gets the same
// values).  With the plan kernel: from its prefix sums and the start-cursor table.
// Without it: the warp loads all context lengths (32 per chunk, every load issued before
// any is used), sums the blocks, and warp 0 scans the chunks to find its start cursor.
struct PieceInfo {
  long long W, pstart, pend;
  int P;
};

__device__ __forceinline__ void piece_setup(const DecodeArgs& a, int p, int P_launch, bool want_cursor, Cursor& cur,
                                            PieceInfo& pi) {
  const int lane = threadIdx.x & 31;
  if (!a.inline_plan) {
    pi.W = (long long)a.n_kv * a.cum[a.batch];
    pi.P = effective_pieces(pi.W, P_launch);
    pi.pstart = pi.W * p / pi.P;
    pi.pend = pi.W * (p + 1) / pi.P;
    if (want_cursor && p < pi.P && pi.pstart < pi.pend) cursor_from_table(cur, p, pi.pstart, a);
    return;
  }
  constexpr int MAXC = kInlinePlanSeqs / 32;
  const int nch = (a.batch + 31) / 32;
  int cv[MAXC];
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    const int s = c * 32 + lane;
    cv[c] = (c < nch && s < a.batch) ? a.ctx_raw[s] : 0;
  }
  long long total = 0;
  bool bad = false;
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    if (c < nch) {
      bad |= cv[c] < 0 || cv[c] > a.max_ctx;
      cv[c] = clamp_ctx(cv[c], a.max_ctx);
      int nb = span_blocks(cv[c], a.window, a.block_size);
#pragma unroll
      for (int o = 16; o; o >>= 1) nb += __shfl_xor_sync(FULL_MASK, nb, o);
      total += nb;
    }
  }
  if (__any_sync(FULL_MASK, bad) && lane == 0 && blockIdx.x == 0 && threadIdx.x == 0) set_err(a.err, PKV_DEV_BAD_CTX);
  pi.W = (long long)a.n_kv * total;
  pi.P = effective_pieces(pi.W, P_launch);
  pi.pstart = pi.W * p / pi.P;
  pi.pend = pi.W * (p + 1) / pi.P;
  if (!want_cursor || p >= pi.P || pi.pstart >= pi.pend) return;
  long long before = 0;                                      // blocks of earlier chunks
  bool found = false;
#pragma unroll
  for (int c = 0; c < MAXC; ++c) {
    if (c >= nch || found) continue;
    const int nb = span_blocks(cv[c], a.window, a.block_size);
    int incl = nb;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += y;
    }
    const long long lo = (long long)a.n_kv * (before + incl - nb), hi = (long long)a.n_kv * (before + incl);
    const unsigned hit = __ballot_sync(FULL_MASK, nb > 0 && lo <= pi.pstart && pi.pstart < hi);
    if (hit) {
      const int src = __ffs(hit) - 1;
      const long long lo_s = __shfl_sync(FULL_MASK, lo, src);
      cur.s = c * 32 + src;
      cur.nb = __shfl_sync(FULL_MASK, nb, src);
      cur.ctx = __shfl_sync(FULL_MASK, cv[c], src);
      cur.b0 = window_first_block(cur.ctx, a.window, a.block_size);
      const long long off = pi.pstart - lo_s;
      cur.g = (int)(off / cur.nb);
      cur.blk = (int)(off % cur.nb);
      cur.seg_start = pi.pstart - cur.blk;
      found = true;
      continue;
    }
    before += __shfl_sync(FULL_MASK, incl, 31);
  }
}

// Advance by one position; only called while positions remain, so a non-empty
// sequence lies ahead when the kv heads of the current one are exhausted.
__device__ __forceinline__ void cursor_next(Cursor& c, const DecodeArgs& a) {
  if (++c.blk < c.nb) return;
  c.seg_start += c.nb;
  c.blk = 0;
  if (++c.g < a.n_kv) return;
  c.g = 0;
  if (a.inline_plan) {
    do {
      ++c.s;
      c.ctx = clamp_ctx(a.ctx_raw[c.s], a.max_ctx);
      c.nb = span_blocks(c.ctx, a.window, a.block_size);
    } while (c.nb == 0 && c.s < a.batch - 1);
  } else {
    do {
      ++c.s;
      c.nb = a.cum[c.s + 1] - a.cum[c.s];
    } while (c.nb == 0 && c.s < a.batch - 1);
    c.ctx = a.ctx_eff[c.s];
  }
  c.b0 = window_first_block(c.ctx, a.window, a.block_size);
}

// One tile's step of the online softmax over tokens (rows of the token-major S^T tiles),
// per head (column), base 2: sc holds the raw scores of TT 16-token tiles x NH 8-head
// tiles in the m16n8 accumulator layout (thread: tokens gid, gid + 8; heads 2*tig + e).
// Scores are scaled, rows outside [lead, ntok) masked, and sc is replaced by the
// exponentials; l and the O^T accumulators are rescaled when the offset rises.
template <int TT, int NH, int MD>
__device__ __forceinline__ void softmax_tile(float (&sc)[TT][NH][4], float (&m)[NH][2], float (&l)[NH][2],
                                             float (&o)[MD][NH][4], int gid, int ntok, int lead, float scale_log2) {
  // Exponents are taken against the running offset m, raised (to the exact running max,
  // with the rescale of l and O) only when a score exceeds it by more than kLazyMax.
  bool over = false;
#pragma unroll
  for (int nh = 0; nh < NH; ++nh)
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int tok = t * 16 + gid + 8 * r;
          float x = sc[t][nh][2 * r + e] * scale_log2;
          if (tok >= ntok || tok < lead) x = -INFINITY;
          sc[t][nh][2 * r + e] = x;
          over |= x > m[nh][e] + kLazyMax;
        }
  if (__any_sync(FULL_MASK, over)) {
#pragma unroll
    for (int nh = 0; nh < NH; ++nh) {
      float al[2];
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float mx = -INFINITY;
#pragma unroll
        for (int t = 0; t < TT; ++t) mx = fmaxf(mx, fmaxf(sc[t][nh][e], sc[t][nh][2 + e]));
        mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 4));
        mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 8));
        mx = fmaxf(mx, __shfl_xor_sync(FULL_MASK, mx, 16));
        const float mn = fmaxf(m[nh][e], mx);
        al[e] = ex2(m[nh][e] - mn);
        m[nh][e] = mn;
        l[nh][e] *= al[e];
      }
#pragma unroll
      for (int md = 0; md < MD; ++md) {
        o[md][nh][0] *= al[0]; o[md][nh][1] *= al[1];
        o[md][nh][2] *= al[0]; o[md][nh][3] *= al[1];
      }
    }
  }
#pragma unroll
  for (int nh = 0; nh < NH; ++nh)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      float rs = 0.f;
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const float pv = ex2(sc[t][nh][2 * r + e] - m[nh][e]);
          sc[t][nh][2 * r + e] = pv;
          rs += pv;
        }
      l[nh][e] += rs;
    }
}

// Records piece p as the first and / or last piece of segment seg (flags of the stage).

// Host launchers (decode_plan.cu).
cudaError_t launch_plan(const int32_t* context_lens, int batch, int max_ctx, int block_size,
                        const DecodeArgs& a, int P, cudaStream_t stream);
// Packing of a tile's row range into the ring's metadata word: rows [lead, ntok) of the
// block are attended (lead > 0 only in a window's first block), plus the F_ flags.
__host__ __device__ __forceinline__ int pack_rows(int ntok, int lead, int flags) {
  return ntok | (flags << 8) | (lead << 16);
}
cudaError_t launch_reduce(int head_dim, const DecodeArgs& a, int P, cudaStream_t stream);
cudaError_t launch_pdl(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args);
int device_sm_count();
// Stages of the shared-memory ring for a stage of `stage_bytes`: about `ring_bytes` of
// ring per CTA, at least 2 and at most 8; the environment variable `env` (an integer
// 2..16) overrides it for tuning.  A small ring leaves room for more resident CTAs,
// which these kernels need more than deep prefetch (the ring sizes each kernel passes
// were measured on the benchmark workloads).
int ring_stages(size_t stage_bytes, size_t ring_bytes, const char* env);
// Head tiling of a group for the attention kernels: 0 = one consumer warp of 8 heads (G <= 8);
// 1 / 2 / 3 = 1 / 2 / 4 warps of 16 heads (G <= 16 / 32 / 64).
inline int head_tiling(int G) { return G <= 8 ? 0 : (G <= 16 ? 1 : (G <= 32 ? 2 : 3)); }
int bf16_pieces(int D, int BS, int G);
// The attention kernel on the fifth-generation tensor cores for groups of 17-32 heads at
// head_dim 128 (decode_tc.cu): its function and dynamic shared memory for a block size.
bool tc_variant(int block_size, const void** fn, size_t* smem);
int int4_pieces(int D, int BS, int G);
void record_cuda_error(cudaError_t e);
int encode_tensor_map_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1);

}  // namespace pkv
