// Paged decode attention over a bf16 cache (GQA / MHA / MQA).
//
// Persistent grid: CTA p streams piece p of the (sequence, kv head, block) line (see
// decode_common.cuh).  A producer walks the piece with a cursor, reads block-table
// entries 32 at a time (and the next 32 ahead), and for each position issues two TMA
// tensor loads per 64-channel box (K and V, 128-byte swizzle) into a ring of `stages`
// shared-memory slots guarded by full/empty mbarriers (for groups of 17-32 heads at block
// size 16, a slot holds two consecutive blocks of a segment).  The producer is a warp of
// its own for groups of up to 32 heads and consumer warp 0 above that.  Consumer warps
// split the group's heads (8 or 16 each), so one K/V read serves every head of the group.
//
// Per block, token-major: S^T = K Q^T with mma.m16n8k16 (the block's tokens on M, heads
// on N; bf16 in, fp32 accumulate; K A-fragments by ldmatrix from the swizzled tile),
// base-2 online softmax over tokens in fp32 with the scale folded in, then
// O^T += V^T P^T with V^T A-fragments by ldmatrix.trans and P^T B-fragments from S^T's
// by an in-register 8x8 transpose; P is split into a bf16 high part and a bf16 low part
// (two mma per tile) so the only rounding of P is below 2^-16 relative.  Segments
// finished inside the piece are normalised and stored; cut segments store (m, l, O)
// partials for the reduce kernel.
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "decode_common.cuh"
#include "nvtx_range.h"

namespace pkv {

template <int D, int BS>
struct Bf16Tile {
  static constexpr int BOX_BYTES = BS * 128;                 // BS rows x 64 channels x 2 B
  static constexpr int NBOX = D / 64;
  static constexpr int TILE = BS * D * 2;                    // one K (or V) tile
  static constexpr int STAGE = 2 * TILE;
};

// TB blocks (K and V tiles each) per ring stage.
template <int D, int BS, int TB>
__host__ __device__ constexpr size_t bf16_smem_bytes(int stages) {
  return 1024 + (size_t)stages * (TB * Bf16Tile<D, BS>::STAGE + 16 + 16);
}

// Keep the halves of a pair of rows (t, t + 1) that lie in [lead, ntok); zero the others.
__device__ __forceinline__ uint32_t mask_pair(uint32_t b, int t, int lead, int ntok) {
  return b & ((t < ntok && t >= lead ? 0x0000ffffu : 0u) | (t + 1 < ntok && t + 1 >= lead ? 0xffff0000u : 0u));
}

// PW: a dedicated producer warp (warp MT) streams the ring ahead of the consumer warps;
// otherwise consumer warp 0 issues each tile's loads itself after consuming a tile.  The
// dedicated warp takes the block-table walk, the barrier bookkeeping and the copy issue
// (about as many cycles per tile as the tile's arithmetic) off the consumers' path; it
// costs one warp of registers, so it is used where the consumers are light (one warp).
// TB = 2: a stage holds two consecutive blocks of one segment when the piece has them, so
// each pass covers 32 token rows at block size 16 (used for groups of 17-32 heads, whose
// consumers spend the most per pass).
template <int D, int BS, int NH, int MT, bool PW, int TB>
__global__ void __launch_bounds__((MT + (PW ? 1 : 0)) * 32,
                                  (PW && BS <= 32) ? (NH == 1 ? 65536 / ((MT + 1) * 32 * 128) : 4) : 0)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const DecodeArgs a) {
  using T = Bf16Tile<D, BS>;
  constexpr int TPB = BS / 16;      // 16-token tiles per block
  constexpr int TT = TB * TPB;      // 16-token tiles per stage
  constexpr int SST = TB * T::STAGE;
  constexpr int KS = D / 16;        // k-steps of K Q^T
  constexpr int MD = D / 16;        // 16-channel m-tiles of O^T
  constexpr int HW = 8 * NH;        // heads per warp
  extern __shared__ uint8_t smem_raw[];
  // aligned by an offset from the array itself, so every access stays a shared-memory one
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int S = a.stages;
  int4* meta = reinterpret_cast<int4*>(smem + (size_t)S * SST);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + S);
  uint64_t* empty = full + S;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tig = lane & 3;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], MT);
    }
    fence_barrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  __syncthreads();
  if (!a.inline_plan) grid_dep_wait();   // the plan kernel's cum / ctx_eff / cursors
  grid_dep_launch();

  const int producer_warp = PW ? MT : 0;
  Cursor cur;
  PieceInfo pi;
  piece_setup(a, blockIdx.x, gridDim.x, warp == producer_warp, cur, pi);
  const int P = pi.P, p = blockIdx.x;
  const long long pstart = pi.pstart, pend = pi.pend;
  const int len = p < P ? (int)(pend - pstart) : 0;
  // A CTA without work still waits for the kernel before it (in inline-plan mode its
  // wait comes below), so no launch after this grid on the stream can pass the append.
  if (len <= 0) {
    if (a.inline_plan) grid_dep_wait();
    return;
  }
  // The setup above reads only this call's inputs; the pools may still be being written by
  // the kernel before this one on the stream (an append launched ahead of the attention),
  // so every thread waits for it here, with the piece's first block-table line on its way.
  if (warp == producer_warp && lane == 0) prefetch_l2(a.bt + (size_t)cur.s * a.max_blocks + cur.b0 + cur.blk);
  if (a.inline_plan) grid_dep_wait();

  // ---------------- producer state (warp-uniform) ----------------
  int w_seq = -1, w_base = 0, w_phys = -1, n_seq = -1, n_base = 0, n_phys = -1;
  const uint64_t pol = policy_evict_first();
  // ring position of the next issue / the next tile consumed (slot, and the parity of the
  // pass over the ring), advanced in order instead of dividing by the stage count
  int p_slot = 0, c_slot = 0;
  uint32_t p_phase = 0, c_phase = 0;

  int pj = 0;                       // next block of the piece to issue (producer warp)
  int issued = 0;                   // stages issued (producer warp)

  // Issues the stage starting at block pj: that block, and with TB = 2 the next one too
  // when it is in the same segment and in the piece.
  auto issue = [&]() {
    if (cur.s != w_seq || cur.blk < w_base || cur.blk >= w_base + 32) {
      if (cur.s == n_seq && cur.blk >= n_base && cur.blk < n_base + 32) {
        w_seq = n_seq; w_base = n_base; w_phys = n_phys;
      } else {
        w_seq = cur.s; w_base = cur.blk;
        const int b = w_base + lane;
        w_phys = b < cur.nb ? __ldg(a.bt + (size_t)cur.s * a.max_blocks + cur.b0 + b) : -1;
      }
      n_seq = cur.s;
      n_base = w_base + 32 < cur.nb ? w_base + 32 : 0;
      const int b = n_base + lane;
      n_phys = b < cur.nb ? __ldg(a.bt + (size_t)cur.s * a.max_blocks + cur.b0 + b) : -1;
    }
    const int phys = __shfl_sync(FULL_MASK, w_phys, cur.blk - w_base);
    const bool pair = TB == 2 && cur.blk + 1 < cur.nb && pj + 1 < len;
    int phys1 = -1;
    if (TB == 2) {
      // the next block's entry is in this window or, past its end, in the prefetched one
      // (which then starts at w_base + 32, as the block is in the segment)
      const int b1 = cur.blk + 1;
      const int x = __shfl_sync(FULL_MASK, w_phys, (b1 - w_base) & 31);
      const int y = __shfl_sync(FULL_MASK, n_phys, (b1 - n_base) & 31);
      phys1 = b1 < w_base + 32 ? x : y;
    }
    const int slot = p_slot;
    const uint32_t ph = p_phase;                               // parity of pass issued / S
    if (++p_slot == S) {
      p_slot = 0;
      p_phase ^= 1u;
    }
    if (lane == 0) {
      bool ok_wait = true;
      if (issued >= S) ok_wait = mbar_wait(&empty[slot], ph ^ 1u);   // released in the previous pass
      if (!ok_wait) {
        set_err(a.err, PKV_DEV_TIMEOUT);
        abort_flag = 1;
      }
      const int nblk = pair ? 2 : 1;
      const int lb = cur.blk + nblk - 1;                       // the stage's last block
      const int ntok = (nblk - 1) * BS + (lb == cur.nb - 1 ? cur.ctx - (cur.b0 + lb) * BS : BS);
      const int lead = cur.blk == 0 ? window_lead(cur.ctx, a.window, BS) : 0;
      const bool end = pj + nblk >= len;
      int flags = 0;
      if (pj == 0 || cur.blk == 0) flags |= F_FIRST;
      if (end || lb == cur.nb - 1) flags |= F_LAST;
      if (cur.seg_start >= pstart && cur.seg_start + cur.nb <= pend) flags |= F_WHOLE;
      if (pair) flags |= F_PAIR;
      if (end) flags |= F_END;
      const bool ok = (unsigned)phys < (unsigned)a.num_blocks && (!pair || (unsigned)phys1 < (unsigned)a.num_blocks);
      if (ok) flags |= F_VALID; else set_err(a.err, PKV_DEV_BAD_BLOCK);
      meta[slot] = make_int4(cur.s, cur.g, cur.blk, pack_rows(ntok, lead, flags));
      if (ok && ok_wait) {
        mbar_arrive_expect_tx(&full[slot], nblk * T::STAGE);
        uint8_t* st = smem + (size_t)slot * SST;
#pragma unroll
        for (int b = 0; b < T::NBOX; ++b) {
          tma_load_3d(st + b * T::BOX_BYTES, &tmk, b * 64, cur.g * BS, phys, &full[slot], pol);
          tma_load_3d(st + T::TILE + b * T::BOX_BYTES, &tmv, b * 64, cur.g * BS, phys, &full[slot], pol);
        }
        if (pair) {
#pragma unroll
          for (int b = 0; b < T::NBOX; ++b) {
            tma_load_3d(st + T::STAGE + b * T::BOX_BYTES, &tmk, b * 64, cur.g * BS, phys1, &full[slot], pol);
            tma_load_3d(st + T::STAGE + T::TILE + b * T::BOX_BYTES, &tmv, b * 64, cur.g * BS, phys1, &full[slot],
                        pol);
          }
        }
      } else {
        mbar_arrive(&full[slot]);
      }
      if (flags & F_FIRST) {                        // warm L2 with the group's queries
        const char* qp = reinterpret_cast<const char*>(a.q) + ((size_t)cur.s * a.n_h + (size_t)cur.g * a.G) * D * 2;
        for (int off = 0; off < a.G * D * 2; off += 128) prefetch_l2(qp + off);
      }
    }
    if (pair) ++cur.blk;                                       // the second block, same segment
    pj += pair ? 2 : 1;
    ++issued;
    if (pj < len) cursor_next(cur, a);
  };

  // ---------------- consumer state (warp w: local heads [w*HW, (w+1)*HW)) ----------------
  // Token-major tiles: S^T[token][head] = K Q^T with the block's tokens on the mma M side
  // and this warp's heads on N (8 per n-tile), then O^T[channel][head] = V^T P^T with
  // P^T's fragments made from S^T's by an in-register 8x8 transpose (movmatrix).
  uint32_t qb[KS][NH][2];
  float o[MD][NH][4];
  float m[NH][2], l[NH][2];
  const int gid = lane >> 2;                    // token row / channel row / head column
  const int hw0 = warp * HW;                    // first local head of this warp

  if (PW && warp == MT) {
    while (pj < len && !abort_flag) issue();
    if (abort_flag && lane == 0) {
      // let the copies still in flight land before the CTA exits: wait (bounded) for the
      // last stage issued on each slot
      for (int k = 0; k < S && k < issued; ++k) {
        const int last = k + ((issued - 1 - k) / S) * S;
        if (!mbar_wait(&full[k], (last / S) & 1)) break;
      }
    }
    return;
  }
  if (!PW && warp == 0)
    for (int k = 0; k < S && pj < len; ++k) issue();

  int consumed = 0;                  // stages consumed
  for (;;) {
    const int slot = c_slot;
    if (!mbar_wait(&full[slot], c_phase) || abort_flag) {
      set_err(a.err, PKV_DEV_TIMEOUT);
      abort_flag = 1;
      break;
    }
    ++consumed;
    const int4 mt = meta[slot];
    const int s = mt.x, g = mt.y, ntok = mt.w & 255, flags = (mt.w >> 8) & 255, lead = mt.w >> 16;
    const size_t qrow0 = (size_t)s * a.n_h + (size_t)g * a.G;   // first q head of the group

    if (flags & F_FIRST) {
#pragma unroll
      for (int nh = 0; nh < NH; ++nh) {
        const int hl = hw0 + nh * 8 + gid;                       // B-fragment column n = gid
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(a.q) + (qrow0 + hl) * (D / 2);
        const bool ok = hl < a.G;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qb[ks][nh][0] = ok ? __ldg(qp + ks * 8 + tig) : 0u;
          qb[ks][nh][1] = ok ? __ldg(qp + ks * 8 + 4 + tig) : 0u;
        }
        m[nh][0] = m[nh][1] = -INFINITY;
        l[nh][0] = l[nh][1] = 0.f;
#pragma unroll
        for (int md = 0; md < MD; ++md) o[md][nh][0] = o[md][nh][1] = o[md][nh][2] = o[md][nh][3] = 0.f;
      }
    }

    if (flags & F_VALID) {
      const uint32_t kb0 = smem_u32(smem + (size_t)slot * SST);   // block k: K at k * STAGE, V after it
      const int nblk = TB > 1 && (flags & F_PAIR) ? 2 : 1;
      // ---- S^T = K Q^T: per 16-token tile and head n-tile, two accumulators (even / odd
      // k-steps) so the dependent mma chains are half as long ----
      float sc[TT][NH][4];
      {
        float sx[TT][NH][4];
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
          for (int nh = 0; nh < NH; ++nh)
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[t][nh][i] = sx[t][nh][i] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
          for (int t = 0; t < TT; ++t) {
            if (t / TPB >= nblk) continue;
            const uint32_t kb = kb0 + (t / TPB) * T::STAGE;
            const int mi = lane >> 3;
            const int tok = (t % TPB) * 16 + ((mi & 1) << 3) + (lane & 7);
            const int ch = 2 * ks + (mi >> 1);
            const uint32_t addr = kb + (ch >> 3) * T::BOX_BYTES + tok * 128 + (((ch & 7) ^ (tok & 7)) << 4);
            uint32_t ka[4];
            ldsm_x4(ka[0], ka[1], ka[2], ka[3], addr);
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
              if (ks & 1) mma_bf16(sx[t][nh], ka, qb[ks][nh][0], qb[ks][nh][1]);
              else mma_bf16(sc[t][nh], ka, qb[ks][nh][0], qb[ks][nh][1]);
            }
          }
        }
#pragma unroll
        for (int t = 0; t < TT; ++t)
#pragma unroll
          for (int nh = 0; nh < NH; ++nh)
#pragma unroll
            for (int i = 0; i < 4; ++i) sc[t][nh][i] += sx[t][nh][i];
      }
      softmax_tile<TT, NH, MD>(sc, m, l, o, gid, ntok, lead, a.scale_log2);
      // ---- O^T += V^T P^T, P as bf16 high + low ----
      const bool partial = ntok < TT * 16 || lead > 0;
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        if (t / TPB >= nblk) continue;
        const uint32_t vb = kb0 + (t / TPB) * T::STAGE + T::TILE;
        // B fragments of P^T (k = token, n = head): the S^T rows of tokens 0-7 / 8-15 of
        // the tile, packed per head pair and transposed
        uint32_t bh[NH][2], bl[NH][2];
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float x = sc[t][nh][2 * r], y = sc[t][nh][2 * r + 1];
            const uint32_t hi = pack_bf16(x, y);
            const uint32_t lo = pack_bf16(x - bf16_lo(hi), y - bf16_hi(hi));
            bh[nh][r] = movmatrix_t(hi);
            bl[nh][r] = movmatrix_t(lo);
          }
        const int t0 = t * 16 + 2 * tig;                   // a0/a1: tokens t0, t0+1; a2/a3: +8
#pragma unroll
        for (int md = 0; md < MD; ++md) {
          const int mi = lane >> 3;
          const int tok = (t % TPB) * 16 + ((mi >> 1) << 3) + (lane & 7);
          const int ch = 2 * md + (mi & 1);
          const uint32_t addr = vb + (ch >> 3) * T::BOX_BYTES + tok * 128 + (((ch & 7) ^ (tok & 7)) << 4);
          uint32_t va[4];
          ldsm_x4_t(va[0], va[1], va[2], va[3], addr);
          if (partial) {
            va[0] = mask_pair(va[0], t0, lead, ntok);
            va[1] = mask_pair(va[1], t0, lead, ntok);
            va[2] = mask_pair(va[2], t0 + 8, lead, ntok);
            va[3] = mask_pair(va[3], t0 + 8, lead, ntok);
          }
#pragma unroll
          for (int nh = 0; nh < NH; ++nh) {
            mma_bf16(o[md][nh], va, bh[nh][0], bh[nh][1]);
            mma_bf16(o[md][nh], va, bl[nh][0], bl[nh][1]);
          }
        }
      }
    }

    if (flags & F_LAST) {
      float L[NH][2];
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x = l[nh][e];
          x += __shfl_xor_sync(FULL_MASK, x, 4);
          x += __shfl_xor_sync(FULL_MASK, x, 8);
          x += __shfl_xor_sync(FULL_MASK, x, 16);
          L[nh][e] = x;
        }
      const bool whole = flags & F_WHOLE;
      const long long part = (long long)s * a.n_kv + g + p;
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hl = hw0 + nh * 8 + 2 * tig + e;           // this thread's head columns
          if (hl >= a.G) continue;
          const float inv = whole ? (L[nh][e] > 0.f ? 1.f / L[nh][e] : 0.f) : 1.f;
          if (whole) {
            const size_t base = (qrow0 + hl) * D;
            if (a.out_f32) {
              float* out = reinterpret_cast<float*>(a.out) + base;
#pragma unroll
              for (int md = 0; md < MD; ++md) {
                out[md * 16 + gid] = o[md][nh][e] * inv;
                out[md * 16 + gid + 8] = o[md][nh][2 + e] * inv;
              }
            } else {
              __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + base;
#pragma unroll
              for (int md = 0; md < MD; ++md) {
                out[md * 16 + gid] = __float2bfloat16_rn(o[md][nh][e] * inv);
                out[md * 16 + gid + 8] = __float2bfloat16_rn(o[md][nh][2 + e] * inv);
              }
            }
          } else {
            float* wo = a.ws_o + ((size_t)part * a.G + hl) * D;
#pragma unroll
            for (int md = 0; md < MD; ++md) {
              wo[md * 16 + gid] = o[md][nh][e];
              wo[md * 16 + gid + 8] = o[md][nh][2 + e];
            }
            if (gid == 0)
              *reinterpret_cast<float2*>(a.ws_ml + ((size_t)part * a.G + hl) * 2) = make_float2(m[nh][e], L[nh][e]);
          }
        }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (!PW && warp == 0 && pj < len) issue();
    if (++c_slot == S) {
      c_slot = 0;
      c_phase ^= 1u;
    }
    if (flags & F_END) break;
  }

  // After a timeout: let this CTA's copies already in flight land before exiting
  // (each wait is bounded, and the drain as a whole gives up at the first failure).
  if (!PW && abort_flag && threadIdx.x == 0) {
    for (int j = consumed; j < issued; ++j)
      if (!mbar_wait(&full[j % S], (j / S) & 1)) break;
  }
}

// ---------------------------------------------------------------------------------------------
struct Bf16Variant {
  const void* fn;
  size_t stage_bytes;
  int stages;
  size_t smem;
  int warps;
  int P;        // persistent CTAs on this device
  bool tc;      // the tensor-memory kernel (takes the query tensor map as well)
};

template <int D, int BS, int NH, int MT, bool PW, int TB>
static Bf16Variant make_variant() {
  Bf16Variant v;
  v.fn = (const void*)decode_bf16_kernel<D, BS, NH, MT, PW, TB>;
  v.stage_bytes = TB * Bf16Tile<D, BS>::STAGE;
  // measured best: 16 KB of ring per CTA with the dedicated producer (its consumer keeps
  // up, and more resident CTAs beat deeper prefetch), 24 KB with the inline one
  v.stages = ring_stages(v.stage_bytes, PW ? 16384 : 24576, "PKV_STAGES_BF16");
  v.smem = bf16_smem_bytes<D, BS, TB>(v.stages);
  v.warps = MT + (PW ? 1 : 0);
  v.P = 0;
  v.tc = false;
  return v;
}

// The tensor-memory kernel (decode_tc.cu) for groups of 17-32 heads at head_dim 128 is taken
// when the environment variable PKV_ATTN_KERNEL is "tc" at the time of the call; by default
// those groups run the mma.sync kernel, measured faster on this shape.
static bool want_tc(int D, int tiling) {
  if (D != 128 || tiling != 2) return false;
  const char* e = getenv("PKV_ATTN_KERNEL");
  return e && e[0] == 't' && e[1] == 'c' && e[2] == 0;
}

static Bf16Variant* lookup_bf16(int D, int BS, int tiling) {
  // One table per process; the library drives one device per process.
  static std::mutex mu;
  static Bf16Variant table[2][3][4][2];
  static bool ready[2][3][4][2] = {};
  const int di = D == 128 ? 1 : 0, bi = BS == 16 ? 0 : (BS == 32 ? 1 : 2), ti = tiling;
  const int tc = want_tc(D, tiling) ? 1 : 0;
  std::lock_guard<std::mutex> lock(mu);
  Bf16Variant& v = table[di][bi][ti][tc];
  if (!ready[di][bi][ti][tc]) {
#define PKV_V(d, b)                                               \
  if (D == d && BS == b) {                                        \
    if (ti == 0) v = make_variant<d, b, 1, 1, true, 1>();         \
    else if (ti == 1) v = make_variant<d, b, 1, 2, true, 1>();    \
    else if (ti == 2) v = make_variant<d, b, 2, 2, true, b == 16 ? 2 : 1>(); \
    else v = make_variant<d, b, 2, 4, false, 1>();                \
  }
    PKV_V(64, 16) PKV_V(64, 32) PKV_V(64, 64) PKV_V(128, 16) PKV_V(128, 32) PKV_V(128, 64)
#undef PKV_V
    // groups of 17-32 heads at head_dim 128 on request: the kernel on the fifth-generation
    // tensor cores (tiles of 128 tokens, accumulators in tensor memory); one CTA of 12 warps per SM
    if (tc) {
      const void* fn = nullptr;
      size_t smem = 0;
      if (tc_variant(BS, &fn, &smem)) {
        v.fn = fn;
        v.smem = smem;
        v.warps = 12;
        v.stages = 2;
        v.stage_bytes = 0;
        v.tc = true;
      }
    }
    if (cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v.smem) != cudaSuccess)
      return nullptr;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, v.fn, v.warps * 32, v.smem) != cudaSuccess || occ < 1)
      return nullptr;
    v.P = device_sm_count() * occ;
    ready[di][bi][ti][tc] = true;
  }
  return &v;
}

int bf16_pieces(int D, int BS, int G) {
  Bf16Variant* v = lookup_bf16(D, BS, head_tiling(G));
  return v ? v->P : 0;
}

}  // namespace pkv

using namespace pkv;

static bool valid_shape(int n_h, int n_kv, int head_dim, int block_size) {
  if (head_dim != 64 && head_dim != 128) return false;
  if (block_size != 16 && block_size != 32 && block_size != 64) return false;
  if (n_kv <= 0 || n_h <= 0 || n_h % n_kv) return false;
  return n_h / n_kv <= 64;
}

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" size_t pkv_decode_workspace_bytes(int batch, int n_h, int n_kv, int head_dim, int block_size, int int4) {
  if (batch < 0 || !valid_shape(n_h, n_kv, head_dim, block_size)) return 0;
  const int G = n_h / n_kv;
  const int P = int4 ? int4_pieces(head_dim, block_size, G) : bf16_pieces(head_dim, block_size, G);
  if (P <= 0) return 0;
  return workspace_layout(batch, n_kv, G, head_dim, P).total;
}

static pkv_status decode_bf16(const void* q, const void* k_pool, const void* v_pool, const int32_t* block_tables,
                              int max_blocks, const int32_t* context_lens, float scale, int window, int batch,
                              int n_h, int n_kv, int head_dim, int block_size, int num_blocks, void* out,
                              int out_dtype, void* workspace, size_t workspace_bytes, int32_t* err_flag,
                              void* stream) {
  if (batch < 0 || !valid_shape(n_h, n_kv, head_dim, block_size) || max_blocks < 0 || num_blocks < 0 || window < 0)
    return PKV_EINVAL;
  if (out_dtype != PKV_OUT_BF16 && out_dtype != PKV_OUT_F32) return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out || !workspace) return PKV_EINVAL;
  if (!al16(q) || !al16(k_pool) || !al16(v_pool) || !al16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_EINVAL;
  if ((long long)max_blocks * block_size > 0x7fffffffLL) return PKV_ERANGE;
  const int G = n_h / n_kv;
  Bf16Variant* v = lookup_bf16(head_dim, block_size, head_tiling(G));
  if (!v) {
    record_cuda_error(cudaGetLastError());
    return PKV_ECUDA;
  }
  const WorkspaceLayout wl = workspace_layout(batch, n_kv, G, head_dim, v->P);
  if (workspace_bytes < wl.total) return PKV_ENOSPC;

  CUtensorMap tmk, tmv;
  const uint64_t rows = (uint64_t)n_kv * block_size;
  const uint64_t row_bytes = (uint64_t)head_dim * 2, block_bytes = rows * row_bytes;
  const uint64_t nblk = num_blocks > 0 ? (uint64_t)num_blocks : 1;
  if (encode_tensor_map_3d(&tmk, k_pool, head_dim, rows, nblk, row_bytes, block_bytes, 64, block_size) ||
      encode_tensor_map_3d(&tmv, v_pool, head_dim, rows, nblk, row_bytes, block_bytes, 64, block_size))
    return PKV_ECUDA;

  char* ws = static_cast<char*>(workspace);
  DecodeArgs a = {};
  a.q = q;
  a.bt = block_tables;
  a.max_blocks = max_blocks;
  a.cum = reinterpret_cast<int32_t*>(ws + wl.cum);
  a.ctx_eff = reinterpret_cast<int32_t*>(ws + wl.ctx);
  a.ctx_raw = context_lens;
  a.max_ctx = max_blocks * block_size;
  a.block_size = block_size;
  a.inline_plan = batch <= kInlinePlanSeqs;
  a.pieces = reinterpret_cast<int4*>(ws + wl.pieces);
  a.P_launch = v->P;
  a.batch = batch;
  a.n_h = n_h;
  a.n_kv = n_kv;
  a.G = G;
  a.num_blocks = num_blocks;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.out = out;
  a.out_f32 = out_dtype == PKV_OUT_F32;
  a.ws_ml = reinterpret_cast<float*>(ws + wl.ml);
  a.ws_o = reinterpret_cast<float*>(ws + wl.o);
  a.err = err_flag;
  a.stages = v->stages;
  a.window = window;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = a.inline_plan ? cudaSuccess
                                : launch_plan(context_lens, batch, max_blocks * block_size, block_size, a, v->P, st);
  if (e == cudaSuccess) {
    if (v->tc) {
      // the group's 32 query rows of a segment, two 64-channel boxes
      CUtensorMap tmq;
      const uint64_t qrows = (uint64_t)batch * n_h;
      if (encode_tensor_map_3d(&tmq, q, 128, qrows, 1, 256, 256 * qrows, 64, 32)) return PKV_ECUDA;
      void* kargs[] = {&tmk, &tmv, &tmq, &a};
      e = launch_pdl(v->fn, dim3(v->P), dim3(v->warps * 32), v->smem, st, kargs);
    } else {
      void* kargs[] = {&tmk, &tmv, &a};
      e = launch_pdl(v->fn, dim3(v->P), dim3(v->warps * 32), v->smem, st, kargs);
    }
  }
  if (e == cudaSuccess) e = launch_reduce(head_dim, a, v->P, st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}

extern "C" pkv_status pkv_paged_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                                            const int32_t* block_tables, int max_blocks,
                                            const int32_t* context_lens, float scale, int batch, int n_h,
                                            int n_kv, int head_dim, int block_size, int num_blocks, void* out,
                                            int out_dtype, void* workspace, size_t workspace_bytes,
                                            int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_paged_decode_attn");
  return decode_bf16(q, k_pool, v_pool, block_tables, max_blocks, context_lens, scale, 0, batch, n_h, n_kv, head_dim,
                     block_size, num_blocks, out, out_dtype, workspace, workspace_bytes, err_flag, stream);
}

extern "C" pkv_status pkv_paged_decode_attn_window(const void* q, const void* k_pool, const void* v_pool,
                                                   const int32_t* block_tables, int max_blocks,
                                                   const int32_t* context_lens, float scale, int window, int batch,
                                                   int n_h, int n_kv, int head_dim, int block_size, int num_blocks,
                                                   void* out, int out_dtype, void* workspace,
                                                   size_t workspace_bytes, int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_paged_decode_attn_window");
  return decode_bf16(q, k_pool, v_pool, block_tables, max_blocks, context_lens, scale, window, batch, n_h, n_kv,
                     head_dim, block_size, num_blocks, out, out_dtype, workspace, workspace_bytes, err_flag, stream);
}

// ---------------------------------------------------------------------------------------------
// Allocation-free variant of pkv_paged_decode_attn.
//
// Some callers cannot allocate device memory at decode time: a serving engine that has
// handed all free device memory to its KV pool up front, a host program that only
// receives device pointers from another runtime which owns the allocator, or code that
// must not call into any allocator on its hot path.  For them the scratch space of the
// decode step lives in a fixed array compiled into this library instead of a
// caller-provided workspace.  The array is PKV_STATIC_SCRATCH_BYTES large and every GPU
// that loads the library holds it until the process exits.
//
// The device address of the array is looked up once per device, on the first call made
// with that device current (host code can only name the array's host-side stand-in);
// make that first call before any stream capture.  Every call shares the one array, so
// calls whose work overlaps on the GPU (different streams, or different host threads)
// race on it and must be serialised by the caller.  Nothing in the array needs to start
// at zero: each call's plan kernel rewrites its prefix sums, and the merge only reads
// partial states the same call wrote.
static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

// The address is kept per device together with the context it was looked up in; after a
// device reset (a new primary context, where the module and its array are loaded again)
// the next call looks it up anew instead of passing a stale address to the kernels.
static void* static_scratch_address() {
  using CtxGetCurrent = CUresult (*)(CUcontext*);
  static CtxGetCurrent ctx_get = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      ctx_get = reinterpret_cast<CtxGetCurrent>(fn);
  });
  static std::mutex mu;
  static void* addr[64] = {};
  static CUcontext owner[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    record_cuda_error(e);
    return nullptr;
  }
  // the context current now (none yet before the runtime's first call on this thread, or
  // right after a reset); the symbol lookup below makes the primary context current
  CUcontext ctx = nullptr;
  if (ctx_get) ctx_get(&ctx);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev] || !ctx || owner[dev] != ctx) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return nullptr;
    }
    CUcontext now = nullptr;
    if (ctx_get) ctx_get(&now);
    addr[dev] = p;
    owner[dev] = now;
  }
  return addr[dev];
}

extern "C" pkv_status pkv_paged_decode_attn_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                                    const int32_t* block_tables, int max_blocks,
                                                    const int32_t* context_lens, float scale, int batch, int n_h,
                                                    int n_kv, int head_dim, int block_size, int num_blocks,
                                                    void* out, int out_dtype, int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_paged_decode_attn_noalloc");
  if (batch < 0 || !valid_shape(n_h, n_kv, head_dim, block_size)) return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  const size_t need = pkv_decode_workspace_bytes(batch, n_h, n_kv, head_dim, block_size, 0);
  if (need == 0) {
    record_cuda_error(cudaGetLastError());
    return PKV_ECUDA;
  }
  if (need > (size_t)PKV_STATIC_SCRATCH_BYTES) return PKV_ERANGE;
  void* ws = static_scratch_address();
  if (!ws) return PKV_ECUDA;
  return pkv_paged_decode_attn(q, k_pool, v_pool, block_tables, max_blocks, context_lens, scale, batch, n_h, n_kv,
                               head_dim, block_size, num_blocks, out, out_dtype, ws, PKV_STATIC_SCRATCH_BYTES,
                               err_flag, stream);
}
