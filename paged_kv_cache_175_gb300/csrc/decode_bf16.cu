// Paged decode attention over a bf16 cache (GQA / MHA / MQA).
//
// Persistent grid: CTA p streams piece p of the (sequence, kv head, block) line (see
// decode_common.cuh).  Warp 0 also acts as the producer: it walks the piece with a
// cursor, reads block-table entries 32 at a time (and the next 32 ahead), and for each
// position issues two TMA tensor loads per tile (K and V, 64-channel boxes with the
// 128-byte swizzle) into a ring of `stages` shared-memory slots guarded by full/empty
// mbarriers.  Each consumer warp owns 16 query heads of the group (an m16 tile; MT
// warps cover the group), so one K/V read serves every head of the group.
//
// Per block: S = Q K^T with mma.m16n8k16 (bf16 in, fp32 accumulate; K B-fragments by
// ldmatrix from the swizzled tile), base-2 online softmax in fp32 with the scale folded
// in, then O += P V with P split into a bf16 high part and a bf16 low part (two mma per
// tile) so the only rounding of P is below 2^-16 relative; V B-fragments by
// ldmatrix.trans.  Segments finished inside the piece are normalised and stored; cut
// segments store (m, l, O) partials for the reduce kernel.
#include <cmath>
#include <mutex>

#include "decode_common.cuh"

namespace pkv {

template <int D, int BS>
struct Bf16Tile {
  static constexpr int BOX_BYTES = BS * 128;                 // BS rows x 64 channels x 2 B
  static constexpr int NBOX = D / 64;
  static constexpr int TILE = BS * D * 2;                    // one K (or V) tile
  static constexpr int STAGE = 2 * TILE;
};

template <int D, int BS>
__host__ __device__ constexpr size_t bf16_smem_bytes(int stages) {
  return 1024 + (size_t)stages * (Bf16Tile<D, BS>::STAGE + 16 + 16);
}

__device__ __forceinline__ uint32_t mask_pair(uint32_t b, int t, int ntok) {
  return b & ((t < ntok ? 0x0000ffffu : 0u) | (t + 1 < ntok ? 0xffff0000u : 0u));
}

template <int D, int BS, int MT>
__global__ void __launch_bounds__(MT * 32)
    decode_bf16_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                       const DecodeArgs a) {
  using T = Bf16Tile<D, BS>;
  constexpr int NT = BS / 8;        // score n-tiles of 8 tokens
  constexpr int KS = D / 16;        // k-steps of Q K^T
  constexpr int DN = D / 8;         // output n-tiles of 8 channels
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  int4* meta = reinterpret_cast<int4*>(smem + (size_t)S * T::STAGE);
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
  grid_dep_wait();                  // plan kernel's cum / ctx_eff are visible after this
  grid_dep_launch();

  const long long W = (long long)a.n_kv * a.cum[a.batch];
  const int P = gridDim.x, p = blockIdx.x;
  const long long pstart = W * p / P, pend = W * (p + 1) / P;
  const int len = (int)(pend - pstart);
  if (len <= 0) return;

  // ---------------- producer state (warp 0, warp-uniform) ----------------
  Cursor cur;
  int w_seq = -1, w_base = 0, w_phys = -1, n_seq = -1, n_base = 0, n_phys = -1;
  const uint64_t pol = policy_evict_first();
  if (warp == 0) cursor_init(cur, pstart, a);

  auto issue = [&](int j) {
    if (cur.s != w_seq || cur.blk < w_base || cur.blk >= w_base + 32) {
      if (cur.s == n_seq && cur.blk >= n_base && cur.blk < n_base + 32) {
        w_seq = n_seq; w_base = n_base; w_phys = n_phys;
      } else {
        w_seq = cur.s; w_base = cur.blk;
        const int b = w_base + lane;
        w_phys = b < cur.nb ? __ldg(a.bt + (size_t)cur.s * a.max_blocks + b) : -1;
      }
      n_seq = cur.s;
      n_base = w_base + 32 < cur.nb ? w_base + 32 : 0;
      const int b = n_base + lane;
      n_phys = b < cur.nb ? __ldg(a.bt + (size_t)cur.s * a.max_blocks + b) : -1;
    }
    const int phys = __shfl_sync(FULL_MASK, w_phys, cur.blk - w_base);
    if (lane == 0) {
      const int slot = j % S;
      bool ok_wait = true;
      if (j >= S) ok_wait = mbar_wait(&empty[slot], ((j / S) - 1) & 1);
      if (!ok_wait) {
        set_err(a.err, PKV_DEV_TIMEOUT);
        abort_flag = 1;
      }
      const int ntok = cur.blk == cur.nb - 1 ? cur.ctx - cur.blk * BS : BS;
      int flags = 0;
      if (j == 0 || cur.blk == 0) flags |= F_FIRST;
      if (j == len - 1 || cur.blk == cur.nb - 1) flags |= F_LAST;
      if (cur.seg_start >= pstart && cur.seg_start + cur.nb <= pend) flags |= F_WHOLE;
      const bool ok = (unsigned)phys < (unsigned)a.num_blocks;
      if (ok) flags |= F_VALID; else set_err(a.err, PKV_DEV_BAD_BLOCK);
      meta[slot] = make_int4(cur.s, cur.g, cur.blk, ntok | (flags << 8));
      if (ok && ok_wait) {
        mbar_arrive_expect_tx(&full[slot], T::STAGE);
        uint8_t* st = smem + (size_t)slot * T::STAGE;
#pragma unroll
        for (int b = 0; b < T::NBOX; ++b) {
          tma_load_3d(st + b * T::BOX_BYTES, &tmk, b * 64, cur.g * BS, phys, &full[slot], pol);
          tma_load_3d(st + T::TILE + b * T::BOX_BYTES, &tmv, b * 64, cur.g * BS, phys, &full[slot], pol);
        }
      } else {
        mbar_arrive(&full[slot]);
      }
      if (flags & F_FIRST) {                        // warm L2 with the group's queries
        const char* qp = reinterpret_cast<const char*>(a.q) + ((size_t)cur.s * a.n_h + (size_t)cur.g * a.G) * D * 2;
        for (int off = 0; off < a.G * D * 2; off += 128) prefetch_l2(qp + off);
      }
    }
    if (j + 1 < len) cursor_next(cur, a);
  };

  // ---------------- consumer state (every warp: 16 heads) ----------------
  uint32_t qa[KS][4];
  float o[DN][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int r0 = lane >> 2;                      // rows r0 and r0 + 8 of the m-tile
  const int hl0 = warp * 16 + r0, hl1 = hl0 + 8; // local head index inside the group
  const bool v0 = hl0 < a.G, v1 = hl1 < a.G;

  if (warp == 0) {
    const int pre = len < S ? len : S;
    for (int j = 0; j < pre; ++j) issue(j);
  }

  int consumed = 0;
  for (int j = 0; j < len; ++j) {
    const int slot = j % S;
    if (!mbar_wait(&full[slot], (j / S) & 1) || abort_flag) {
      set_err(a.err, PKV_DEV_TIMEOUT);
      abort_flag = 1;
      break;
    }
    consumed = j + 1;
    const int4 mt = meta[slot];
    const int s = mt.x, g = mt.y, ntok = mt.w & 255, flags = mt.w >> 8;

    if (flags & F_FIRST) {
      const uint32_t* q0 = reinterpret_cast<const uint32_t*>(a.q) + ((size_t)s * a.n_h + (size_t)g * a.G + hl0) * (D / 2);
      const uint32_t* q1 = q0 + 8 * (D / 2);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = v0 ? __ldg(q0 + ks * 8 + tig) : 0u;
        qa[ks][1] = v1 ? __ldg(q1 + ks * 8 + tig) : 0u;
        qa[ks][2] = v0 ? __ldg(q0 + ks * 8 + 4 + tig) : 0u;
        qa[ks][3] = v1 ? __ldg(q1 + ks * 8 + 4 + tig) : 0u;
      }
#pragma unroll
      for (int n = 0; n < DN; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
    }

    if (flags & F_VALID) {
      const uint32_t kb = smem_u32(smem + (size_t)slot * T::STAGE), vb = kb + T::TILE;
      float sc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
      // S = Q K^T
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
        for (int np = 0; np < NT / 2; ++np) {
          const int tok = np * 16 + ((lane >> 4) << 3) + (lane & 7);
          const int ch = 2 * ks + ((lane >> 3) & 1);
          const uint32_t addr = kb + (ch >> 3) * T::BOX_BYTES + tok * 128 + (((ch & 7) ^ (tok & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3, addr);
          mma_bf16(sc[2 * np], qa[ks], b0, b1);
          mma_bf16(sc[2 * np + 1], qa[ks], b2, b3);
        }
      }
      // online softmax (base 2)
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = n * 8 + 2 * tig + e;
          float x0 = sc[n][e] * a.scale_log2, x1 = sc[n][2 + e] * a.scale_log2;
          if (tok >= ntok) x0 = x1 = -INFINITY;
          sc[n][e] = x0;
          sc[n][2 + e] = x1;
          mx0 = fmaxf(mx0, x0);
          mx1 = fmaxf(mx1, x1);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(FULL_MASK, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(FULL_MASK, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = ex2(m0 - mn0), al1 = ex2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sc[n][e] = ex2(sc[n][e] - mn0);
          sc[n][2 + e] = ex2(sc[n][2 + e] - mn1);
          rs0 += sc[n][e];
          rs1 += sc[n][2 + e];
        }
      }
      l0 = l0 * al0 + rs0;
      l1 = l1 * al1 + rs1;
      if (__any_sync(FULL_MASK, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
        for (int n = 0; n < DN; ++n) {
          o[n][0] *= al0; o[n][1] *= al0; o[n][2] *= al1; o[n][3] *= al1;
        }
      }
      // O += P V, P as bf16 high + low
      const bool partial = ntok < BS;
#pragma unroll
      for (int kt = 0; kt < BS / 16; ++kt) {
        uint32_t ah[4], al[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x = sc[2 * kt + (i >> 1)][(i & 1) * 2], y = sc[2 * kt + (i >> 1)][(i & 1) * 2 + 1];
          ah[i] = pack_bf16(x, y);
          al[i] = pack_bf16(x - bf16_lo(ah[i]), y - bf16_hi(ah[i]));
        }
        const int t0 = kt * 16 + 2 * tig;
#pragma unroll
        for (int nb = 0; nb < D / 16; ++nb) {
          const int tok = kt * 16 + (((lane >> 3) & 1) << 3) + (lane & 7);
          const int ch = 2 * nb + (lane >> 4);
          const uint32_t addr = vb + (ch >> 3) * T::BOX_BYTES + tok * 128 + (((ch & 7) ^ (tok & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, addr);
          if (partial) {
            b0 = mask_pair(b0, t0, ntok);
            b2 = mask_pair(b2, t0, ntok);
            b1 = mask_pair(b1, t0 + 8, ntok);
            b3 = mask_pair(b3, t0 + 8, ntok);
          }
          mma_bf16(o[2 * nb], ah, b0, b1);
          mma_bf16(o[2 * nb], al, b0, b1);
          mma_bf16(o[2 * nb + 1], ah, b2, b3);
          mma_bf16(o[2 * nb + 1], al, b2, b3);
        }
      }
    }

    if (flags & F_LAST) {
      float L0 = l0 + __shfl_xor_sync(FULL_MASK, l0, 1);
      L0 += __shfl_xor_sync(FULL_MASK, L0, 2);
      float L1 = l1 + __shfl_xor_sync(FULL_MASK, l1, 1);
      L1 += __shfl_xor_sync(FULL_MASK, L1, 2);
      if (flags & F_WHOLE) {
        const float i0 = L0 > 0.f ? 1.f / L0 : 0.f, i1 = L1 > 0.f ? 1.f / L1 : 0.f;
        const size_t row0 = (size_t)s * a.n_h + (size_t)g * a.G + hl0;
        if (a.out_f32) {
          float* out0 = reinterpret_cast<float*>(a.out) + row0 * D;
          float* out1 = out0 + 8 * D;
#pragma unroll
          for (int n = 0; n < DN; ++n) {
            if (v0) *reinterpret_cast<float2*>(out0 + n * 8 + 2 * tig) = make_float2(o[n][0] * i0, o[n][1] * i0);
            if (v1) *reinterpret_cast<float2*>(out1 + n * 8 + 2 * tig) = make_float2(o[n][2] * i1, o[n][3] * i1);
          }
        } else {
          uint32_t* out0 = reinterpret_cast<uint32_t*>(a.out) + row0 * (D / 2);
          uint32_t* out1 = out0 + 8 * (D / 2);
#pragma unroll
          for (int n = 0; n < DN; ++n) {
            if (v0) out0[n * 4 + tig] = pack_bf16(o[n][0] * i0, o[n][1] * i0);
            if (v1) out1[n * 4 + tig] = pack_bf16(o[n][2] * i1, o[n][3] * i1);
          }
        }
      } else {
        const long long part = (long long)s * a.n_kv + g + p;
        float* wo = a.ws_o + (size_t)part * a.G * D;
#pragma unroll
        for (int n = 0; n < DN; ++n) {
          if (v0) *reinterpret_cast<float2*>(wo + (size_t)hl0 * D + n * 8 + 2 * tig) = make_float2(o[n][0], o[n][1]);
          if (v1) *reinterpret_cast<float2*>(wo + (size_t)hl1 * D + n * 8 + 2 * tig) = make_float2(o[n][2], o[n][3]);
        }
        if (tig == 0) {
          if (v0) *reinterpret_cast<float2*>(a.ws_ml + ((size_t)part * a.G + hl0) * 2) = make_float2(m0, L0);
          if (v1) *reinterpret_cast<float2*>(a.ws_ml + ((size_t)part * a.G + hl1) * 2) = make_float2(m1, L1);
        }
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (warp == 0 && j + S < len) issue(j + S);
  }

  // After a timeout: let this CTA's copies already in flight land before exiting
  // (each wait is bounded, and the drain as a whole gives up at the first failure).
  if (abort_flag && threadIdx.x == 0) {
    const int issued = len < consumed + S ? len : consumed + S;
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
};

template <int D, int BS, int MT>
static Bf16Variant make_variant() {
  Bf16Variant v;
  v.fn = (const void*)decode_bf16_kernel<D, BS, MT>;
  v.stage_bytes = Bf16Tile<D, BS>::STAGE;
  v.stages = ring_stages(v.stage_bytes, "PKV_STAGES_BF16");
  v.smem = bf16_smem_bytes<D, BS>(v.stages);
  v.warps = MT;
  v.P = 0;
  return v;
}

int mt_for_group(int G) { return G <= 16 ? 1 : (G <= 32 ? 2 : 4); }

static Bf16Variant* lookup_bf16(int D, int BS, int MT) {
  // One table per process; the library drives one device per process.
  static std::mutex mu;
  static Bf16Variant table[2][3][3];
  static bool ready[2][3][3] = {};
  const int di = D == 128 ? 1 : 0, bi = BS == 16 ? 0 : (BS == 32 ? 1 : 2), mi = MT == 1 ? 0 : (MT == 2 ? 1 : 2);
  std::lock_guard<std::mutex> lock(mu);
  Bf16Variant& v = table[di][bi][mi];
  if (!ready[di][bi][mi]) {
#define PKV_V(d, b, m) \
  if (D == d && BS == b && MT == m) v = make_variant<d, b, m>();
    PKV_V(64, 16, 1) PKV_V(64, 16, 2) PKV_V(64, 16, 4)
    PKV_V(64, 32, 1) PKV_V(64, 32, 2) PKV_V(64, 32, 4)
    PKV_V(64, 64, 1) PKV_V(64, 64, 2) PKV_V(64, 64, 4)
    PKV_V(128, 16, 1) PKV_V(128, 16, 2) PKV_V(128, 16, 4)
    PKV_V(128, 32, 1) PKV_V(128, 32, 2) PKV_V(128, 32, 4)
    PKV_V(128, 64, 1) PKV_V(128, 64, 2) PKV_V(128, 64, 4)
#undef PKV_V
    if (cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v.smem) != cudaSuccess)
      return nullptr;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, v.fn, v.warps * 32, v.smem) != cudaSuccess || occ < 1)
      return nullptr;
    v.P = device_sm_count() * occ;
    ready[di][bi][mi] = true;
  }
  return &v;
}

int bf16_pieces(int D, int BS, int G) {
  Bf16Variant* v = lookup_bf16(D, BS, mt_for_group(G));
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

extern "C" pkv_status pkv_paged_decode_attn(const void* q, const void* k_pool, const void* v_pool,
                                            const int32_t* block_tables, int max_blocks,
                                            const int32_t* context_lens, float scale, int batch, int n_h,
                                            int n_kv, int head_dim, int block_size, int num_blocks, void* out,
                                            int out_dtype, void* workspace, size_t workspace_bytes,
                                            int32_t* err_flag, void* stream) {
  if (batch < 0 || !valid_shape(n_h, n_kv, head_dim, block_size) || max_blocks < 0 || num_blocks < 0)
    return PKV_EINVAL;
  if (out_dtype != PKV_OUT_BF16 && out_dtype != PKV_OUT_F32) return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  if (!q || !k_pool || !v_pool || !block_tables || !context_lens || !out || !workspace) return PKV_EINVAL;
  if (!al16(q) || !al16(k_pool) || !al16(v_pool) || !al16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_EINVAL;
  if ((long long)max_blocks * block_size > 0x7fffffffLL) return PKV_ERANGE;
  const int G = n_h / n_kv, MT = mt_for_group(G);
  Bf16Variant* v = lookup_bf16(head_dim, block_size, MT);
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

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_plan(context_lens, batch, max_blocks * block_size, block_size, a, st);
  if (e == cudaSuccess) {
    void* kargs[] = {&tmk, &tmv, &a};
    e = launch_pdl(v->fn, dim3(v->P), dim3(v->warps * 32), v->smem, st, kargs);
  }
  if (e == cudaSuccess) e = launch_reduce(head_dim, a, v->P, st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
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

static void* static_scratch_address() {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64) {
    record_cuda_error(e);
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

extern "C" pkv_status pkv_paged_decode_attn_noalloc(const void* q, const void* k_pool, const void* v_pool,
                                                    const int32_t* block_tables, int max_blocks,
                                                    const int32_t* context_lens, float scale, int batch, int n_h,
                                                    int n_kv, int head_dim, int block_size, int num_blocks,
                                                    void* out, int out_dtype, int32_t* err_flag, void* stream) {
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
