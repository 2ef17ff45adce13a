// INT4 paged KV cache: quantize-on-append and decode attention with in-register
// dequantization.  Format and exact quantizer op sequence are documented in pkv.h.
#include <cmath>
#include <mutex>

#include "decode_common.cuh"

namespace pkv {

// nibble index (0..7) inside a 32-bit word of the code row that holds channel c' (0..7)
__host__ __device__ constexpr int nibble_of(int c) { return (c & 1) ? 4 + (c >> 1) : (c >> 1); }
// channel offset held by nibble n
__host__ __device__ constexpr int channel_of(int n) { return n < 4 ? 2 * n : 2 * (n - 4) + 1; }

struct GroupQuant {
  float s, m;           // fp16 scale / min, widened
  __half s16, m16;
};

// Steps (1)-(3) of the quantizer: fp32 range, fp32 step, fp16 scale and min.
// A zero minimum is stored as +0.
__device__ __forceinline__ GroupQuant group_params(float lo, float hi) {
  if (lo == 0.f) lo = 0.f;
  GroupQuant q;
  const float s32 = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
  q.s16 = __float2half_rn(s32);
  q.m16 = __float2half_rn(lo);
  q.s = __half2float(q.s16);
  q.m = __half2float(q.m16);
  return q;
}
// Step (4): code of one value.
__device__ __forceinline__ uint32_t quant_code(float x, const GroupQuant& q) {
  if (q.s == 0.f) return 0u;
  float c = rintf(__fdiv_rn(__fsub_rn(x, q.m), q.s));
  c = fminf(fmaxf(c, 0.f), 15.f);
  return (uint32_t)c;
}

__device__ __forceinline__ float warp_min(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fminf(x, __shfl_xor_sync(FULL_MASK, x, o));
  return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o; o >>= 1) x = fmaxf(x, __shfl_xor_sync(FULL_MASK, x, o));
  return x;
}

struct QuantAppendArgs {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const int64_t* slots;
  const int32_t* tail_seq;
  int n_tok, n_kv, block_size, tail_rows;
  long long n_slots;
  uint8_t* k_codes;
  __half* k_meta;
  uint8_t* v_codes;
  __half* v_meta;
  __nv_bfloat16* k_tail;
  int32_t* err;
};

// Phase 1: one warp per (token, kv head).  V is quantized per token; a token that fills
// the last row of its block also quantizes that block's K per channel, taking rows
// appended earlier in this call from `k` and older rows from the tail.
template <int D>
__global__ void __launch_bounds__(256) quant_append_kernel(const QuantAppendArgs a) {
  constexpr int CPL = D / 32;                   // V channels per lane
  constexpr int LPW = 8 / CPL;                  // lanes per 32-bit code word
  const int lane = threadIdx.x & 31;
  const long long wid = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  if (wid >= (long long)a.n_tok * a.n_kv) return;
  const int i = (int)(wid / a.n_kv), g = (int)(wid % a.n_kv);
  const long long slot = a.slots[i];
  if (slot < 0) return;
  const int seq = a.tail_seq[i];
  if (slot >= a.n_slots || (unsigned)seq >= (unsigned)a.tail_rows) {
    if (lane == 0 && g == 0) set_err(a.err, PKV_DEV_BAD_SLOT);
    return;
  }
  const int BS = a.block_size;
  const long long blk = slot / BS;
  const int row = (int)(slot - blk * BS);
  const size_t tile = (size_t)blk * a.n_kv + g;           // (block, kv head)

  // ---- V: per token ----
  {
    const __nv_bfloat16* src = a.v + ((size_t)i * a.n_kv + g) * D + lane * CPL;
    float x[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) x[c] = __bfloat162float(src[c]);
    float lo = x[0], hi = x[0];
#pragma unroll
    for (int c = 1; c < CPL; ++c) { lo = fminf(lo, x[c]); hi = fmaxf(hi, x[c]); }
    lo = warp_min(lo);
    hi = warp_max(hi);
    const GroupQuant q = group_params(lo, hi);
    uint32_t word = 0;
#pragma unroll
    for (int c = 0; c < CPL; ++c) {
      const int ch = (lane * CPL + c) & 7;
      word |= quant_code(x[c], q) << (4 * nibble_of(ch));
    }
#pragma unroll
    for (int o = 1; o < LPW; o <<= 1) word |= __shfl_xor_sync(FULL_MASK, word, o);
    uint32_t* dst = reinterpret_cast<uint32_t*>(a.v_codes + (tile * BS + row) * (D / 2));
    if (lane % LPW == 0) dst[lane / LPW] = word;
    if (lane == 0) {
      __half2 meta = __halves2half2(q.s16, q.m16);
      reinterpret_cast<__half2*>(a.v_meta)[tile * BS + row] = meta;
    }
  }

  // ---- K: only the token that fills the block ----
  if (row != BS - 1) return;
  // rows [BS-1-run, BS-1] come from this call (tokens i-run .. i), the rest from the tail
  int run = 0;
  for (int base = 1; base < BS; base += 32) {
    const int kk = base + lane;
    bool ok = true;
    if (kk < BS) {
      const int j = i - kk;
      ok = j >= 0 && a.slots[j] == slot - kk && a.tail_seq[j] == seq;
    }
    const unsigned bad = __ballot_sync(FULL_MASK, !ok);
    if (bad) {
      run += __ffs(bad) - 1;
      break;
    }
    run += 32 < BS - base ? 32 : BS - base;
  }
  const int first_call_row = BS - 1 - run;
  const __nv_bfloat16* krow_call = a.k + g * D;            // token t: + t * n_kv * D
  const __nv_bfloat16* krow_tail = a.k_tail + ((size_t)seq * a.n_kv + g) * BS * D;
  __half* kmeta = a.k_meta + tile * 2 * D;
  uint32_t* kcodes = reinterpret_cast<uint32_t*>(a.k_codes + tile * BS * (D / 2));
#pragma unroll 1
  for (int cm = 0; cm < CPL; ++cm) {
    const int c = lane + 32 * cm;                            // this lane's channel
    auto val = [&](int r) -> float {
      const __nv_bfloat16* p = r >= first_call_row ? krow_call + (size_t)(i - (BS - 1 - r)) * a.n_kv * D
                                                   : krow_tail + (size_t)r * D;
      return __bfloat162float(p[c]);
    };
    float lo = val(0), hi = lo;
    for (int r = 1; r < BS; ++r) {
      const float x = val(r);
      lo = fminf(lo, x);
      hi = fmaxf(hi, x);
    }
    const GroupQuant q = group_params(lo, hi);
    kmeta[c] = q.s16;
    kmeta[D + c] = q.m16;
    for (int r = 0; r < BS; ++r) {
      uint32_t word = quant_code(val(r), q) << (4 * nibble_of(c & 7));
      word |= __shfl_xor_sync(FULL_MASK, word, 1);
      word |= __shfl_xor_sync(FULL_MASK, word, 2);
      word |= __shfl_xor_sync(FULL_MASK, word, 4);
      if ((lane & 7) == 0) kcodes[(size_t)r * (D / 8) + c / 8] = word;
    }
  }
}

// Phase 2: K rows of blocks that stay unfinished after this call go to the tail.
template <int D>
__global__ void __launch_bounds__(256) tail_write_kernel(const QuantAppendArgs a) {
  constexpr int VEC = D / 8;                                 // 16-byte vectors per row
  const long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  if (idx >= (long long)a.n_tok * a.n_kv * VEC) return;
  const int vec = (int)(idx % VEC);
  const long long rowid = idx / VEC;
  const int i = (int)(rowid / a.n_kv), g = (int)(rowid % a.n_kv);
  const long long slot = a.slots[i];
  if (slot < 0 || slot >= a.n_slots) return;                // bad slots were flagged in phase 1
  const int seq = a.tail_seq[i];
  if ((unsigned)seq >= (unsigned)a.tail_rows) return;
  const int BS = a.block_size;
  const int row = (int)(slot % BS);
  const int ahead = BS - 1 - row;                            // the block's last row is token i + ahead
  const int j = i + ahead;
  if (j < a.n_tok && a.slots[j] == slot + ahead && a.tail_seq[j] == seq) return;
  const uint4* src = reinterpret_cast<const uint4*>(a.k + ((size_t)i * a.n_kv + g) * D) + vec;
  uint4* dst = reinterpret_cast<uint4*>(a.k_tail + (((size_t)seq * a.n_kv + g) * BS + row) * D) + vec;
  *dst = *src;
}

// ---------------------------------------------------------------------------------------------
// Decode attention over the INT4 cache.
//
// Stage layout for one (block, kv head): K codes [BS][D/2], V codes [BS][D/2], K meta
// [2][D] fp16, V meta [BS][2] fp16, and room for a bf16 K tail [BS][D] used only by a
// sequence's unfinished last block.  Each piece is one 1-D bulk copy.
//
// Q K^T uses fp16 mma.  The channel order inside a k-step is chosen so each thread's
// B-fragment comes from one 16-byte load of its token row: thread t of a quad owns
// channels [t*D/4, (t+1)*D/4); k-step ks takes word ks/2 and, inside it, channel pairs
// (0,1),(2,3) or (4,5),(6,7).  The A-fragment (q, converted to fp16 once per segment
// part) uses the same channel order.  Dequantization x^ = fp16(code * s + m) runs on
// half2 pairs: the code pair is unpacked into 1024 + code by a mask-and-or, 1024 is
// subtracted (exact), then one fused multiply-add with the channel pair's (s, m) rounds
// the exact value once, as the format defines it.
//
// P V uses fp16 mma with P carried as an fp16 high part plus an fp16 low part (two mma
// per tile).  Thread u of a group of four owns output channels [u*D/8, (u+1)*D/8) as
// B-fragment columns; a byte of a V code word pairs the same nibble of two token rows
// (byte permute), giving a half2 of two tokens of one channel, scaled by the two
// tokens' (s, m).
template <int D, int BS>
struct Int4Tile {
  static constexpr int KC = 0;
  static constexpr int VC = BS * D / 2;
  static constexpr int KM = BS * D;
  static constexpr int VM = BS * D + 4 * D;
  static constexpr int KT = (BS * D + 4 * D + 4 * BS + 15) / 16 * 16;
  static constexpr int STAGE = (KT + BS * D * 2 + 127) / 128 * 128;
  static constexpr int FULL_BYTES = BS * D + 4 * D + 4 * BS;          // codes + metadata
  static constexpr int TAIL_BYTES = BS * D / 2 + 4 * BS + 2 * BS * D;   // V codes + V meta + K tail
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t lop_nib(uint32_t x) {   // (x & 0x000f000f) | 0x64006400
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(d) : "r"(x), "r"(0x000f000fu), "r"(0x64006400u));
  return d;
}
__device__ __forceinline__ uint32_t dq2(uint32_t h1024, uint32_t s2, uint32_t m2) {
  const __half2 c = __hsub2(*reinterpret_cast<const __half2*>(&h1024), __half2half2(__ushort_as_half(0x6400)));
  const __half2 r = __hfma2(c, *reinterpret_cast<const __half2*>(&s2), *reinterpret_cast<const __half2*>(&m2));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) { return pack_f16(bf16_lo(w), bf16_hi(w)); }

template <int D, int BS>
__host__ __device__ constexpr size_t int4_smem_bytes(int stages) {
  return 1024 + (size_t)stages * (Int4Tile<D, BS>::STAGE + 16 + 16);
}

template <int D, int BS, int MT>
__global__ void __launch_bounds__(MT * 32) decode_int4_kernel(const DecodeArgs a) {
  using T = Int4Tile<D, BS>;
  constexpr int NT = BS / 8;
  constexpr int KS = D / 16;
  constexpr int DN = D / 8;
  constexpr int KW = D / 32;        // K code words per thread per token row
  constexpr int CB = D / 4;         // K channels per thread (QK k-slots)
  constexpr int CV = D / 8;         // V channels per thread (PV columns)
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int S = a.stages;
  int4* meta = reinterpret_cast<int4*>(smem + (size_t)S * T::STAGE);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + S);
  uint64_t* empty = full + S;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tig = lane & 3, u = lane >> 2;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], MT);
    }
    fence_barrier_init();
  }
  __syncthreads();
  grid_dep_wait();
  grid_dep_launch();

  Cursor cur;
  PieceInfo pi;
  piece_setup(a, blockIdx.x, gridDim.x, warp == 0, cur, pi);
  const int P = pi.P, p = blockIdx.x;
  if (p >= P) return;
  const long long pstart = pi.pstart, pend = pi.pend;
  const int len = (int)(pend - pstart);
  if (len <= 0) return;

  int w_seq = -1, w_base = 0, w_phys = -1, n_seq = -1, n_base = 0, n_phys = -1;
  const uint64_t pol = policy_evict_first();

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
        uint8_t* st = smem + (size_t)slot * T::STAGE;
        const size_t tile = (size_t)phys * a.n_kv + cur.g;
        if (ntok == BS) {
          mbar_arrive_expect_tx(&full[slot], T::FULL_BYTES);
          bulk_g2s(st + T::KC, a.k_codes + tile * (BS * D / 2), BS * D / 2, &full[slot], pol);
          bulk_g2s(st + T::VC, a.v_codes + tile * (BS * D / 2), BS * D / 2, &full[slot], pol);
          bulk_g2s(st + T::KM, a.k_meta + tile * (2 * D), 4 * D, &full[slot], pol);
          bulk_g2s(st + T::VM, a.v_meta + tile * (2 * BS), 4 * BS, &full[slot], pol);
        } else {
          mbar_arrive_expect_tx(&full[slot], T::TAIL_BYTES);
          bulk_g2s(st + T::VC, a.v_codes + tile * (BS * D / 2), BS * D / 2, &full[slot], pol);
          bulk_g2s(st + T::VM, a.v_meta + tile * (2 * BS), 4 * BS, &full[slot], pol);
          bulk_g2s(st + T::KT, a.k_tail + ((size_t)cur.s * a.n_kv + cur.g) * BS * D, 2 * BS * D, &full[slot], pol);
        }
      } else {
        mbar_arrive(&full[slot]);
      }
      if (flags & F_FIRST) {
        const char* qp = reinterpret_cast<const char*>(a.q) + ((size_t)cur.s * a.n_h + (size_t)cur.g * a.G) * D * 2;
        for (int off = 0; off < a.G * D * 2; off += 128) prefetch_l2(qp + off);
      }
    }
    if (j + 1 < len) cursor_next(cur, a);
  };

  uint32_t qa[KS][4];
  float o[DN][4];
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  const int hl0 = warp * 16 + u, hl1 = hl0 + 8;
  const bool v0 = hl0 < a.G, v1 = hl1 < a.G;
  const int cb = tig * CB;           // first K channel of this thread
  const int cv = u * CV;             // first V output column channel of this thread

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
        const int w = (cb + 8 * (ks >> 1) + 4 * (ks & 1)) >> 1;   // word of channel pair (c0, c0+1)
        qa[ks][0] = v0 ? bf2_to_h2(__ldg(q0 + w)) : 0u;
        qa[ks][1] = v1 ? bf2_to_h2(__ldg(q1 + w)) : 0u;
        qa[ks][2] = v0 ? bf2_to_h2(__ldg(q0 + w + 1)) : 0u;
        qa[ks][3] = v1 ? bf2_to_h2(__ldg(q1 + w + 1)) : 0u;
      }
#pragma unroll
      for (int n = 0; n < DN; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
    }

    if (flags & F_VALID) {
      const uint8_t* st = smem + (size_t)slot * T::STAGE;
      const bool tailblk = ntok < BS;
      float sc[NT][4];
#pragma unroll
      for (int n = 0; n < NT; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
      // ---- S = Q K^T ----
      if (!tailblk) {
        uint32_t s2[CB / 2], m2[CB / 2];                          // (s, m) of channel pairs cb + 2k
        const uint4* kms = reinterpret_cast<const uint4*>(st + T::KM + cb * 2);
        const uint4* kmm = reinterpret_cast<const uint4*>(st + T::KM + 2 * D + cb * 2);
#pragma unroll
        for (int k4 = 0; k4 < CB / 8; ++k4) {
          const uint4 a4 = kms[k4], b4 = kmm[k4];
          s2[4 * k4] = a4.x; s2[4 * k4 + 1] = a4.y; s2[4 * k4 + 2] = a4.z; s2[4 * k4 + 3] = a4.w;
          m2[4 * k4] = b4.x; m2[4 * k4 + 1] = b4.y; m2[4 * k4 + 2] = b4.z; m2[4 * k4 + 3] = b4.w;
        }
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          uint32_t wd[KW];
          const uint8_t* rowp = st + T::KC + (n * 8 + u) * (D / 2) + tig * (D / 8);
          if constexpr (KW == 4) {
            const uint4 t4 = *reinterpret_cast<const uint4*>(rowp);
            wd[0] = t4.x; wd[1] = t4.y; wd[2] = t4.z; wd[3] = t4.w;
          } else {
            const uint2 t2 = *reinterpret_cast<const uint2*>(rowp);
            wd[0] = t2.x; wd[1] = t2.y;
          }
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int w = ks >> 1, hsel = 2 * (ks & 1);         // pairs h_hsel, h_hsel+1 of word w
            const uint32_t x0 = lop_nib(wd[w] >> (4 * hsel)), x1 = lop_nib(wd[w] >> (4 * hsel + 4));
            const int pr = 4 * w + hsel;                         // channel pair index (cb + 2*pr)
            const uint32_t b0 = dq2(x0, s2[pr], m2[pr]), b1 = dq2(x1, s2[pr + 1], m2[pr + 1]);
            mma_f16(sc[n], qa[ks], b0, b1);
          }
        }
      } else {
#pragma unroll
        for (int n = 0; n < NT; ++n) {
          const uint4* rowp = reinterpret_cast<const uint4*>(st + T::KT + (size_t)(n * 8 + u) * D * 2 + cb * 2);
          uint32_t wd[CB / 2];
#pragma unroll
          for (int k4 = 0; k4 < CB / 8; ++k4) {
            const uint4 t4 = rowp[k4];
            wd[4 * k4] = t4.x; wd[4 * k4 + 1] = t4.y; wd[4 * k4 + 2] = t4.z; wd[4 * k4 + 3] = t4.w;
          }
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int pr = 4 * (ks >> 1) + 2 * (ks & 1);
            mma_f16(sc[n], qa[ks], bf2_to_h2(wd[pr]), bf2_to_h2(wd[pr + 1]));
          }
        }
      }
      // ---- online softmax (base 2) ----
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
      // ---- O += P V ----
      const uint32_t* vm = reinterpret_cast<const uint32_t*>(st + T::VM);
#pragma unroll
      for (int kt = 0; kt < BS / 16; ++kt) {
        uint32_t pa[4], pl[4];                                    // P = high + low, both fp16
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float x = sc[2 * kt + (i >> 1)][(i & 1) * 2], y = sc[2 * kt + (i >> 1)][(i & 1) * 2 + 1];
          pa[i] = pack_f16(x, y);
          const __half2 h = *reinterpret_cast<const __half2*>(&pa[i]);
          pl[i] = pack_f16(x - __low2float(h), y - __high2float(h));
        }
        const int t0 = kt * 16 + 2 * tig;                        // b0: tokens t0, t0+1; b1: t0+8, t0+9
        const uint32_t sA = prmt(vm[t0], vm[t0 + 1], 0x5410), mA = prmt(vm[t0], vm[t0 + 1], 0x7632);
        const uint32_t sB = prmt(vm[t0 + 8], vm[t0 + 9], 0x5410), mB = prmt(vm[t0 + 8], vm[t0 + 9], 0x7632);
        const uint8_t* vc = st + T::VC + cv / 2;
        uint32_t ra[CV / 8], rb[CV / 8], rc[CV / 8], rd[CV / 8];   // code words of rows t0, t0+1, t0+8, t0+9
#pragma unroll
        for (int w = 0; w < CV / 8; ++w) {
          ra[w] = *reinterpret_cast<const uint32_t*>(vc + (size_t)t0 * (D / 2) + 4 * w);
          rb[w] = *reinterpret_cast<const uint32_t*>(vc + (size_t)(t0 + 1) * (D / 2) + 4 * w);
          rc[w] = *reinterpret_cast<const uint32_t*>(vc + (size_t)(t0 + 8) * (D / 2) + 4 * w);
          rd[w] = *reinterpret_cast<const uint32_t*>(vc + (size_t)(t0 + 9) * (D / 2) + 4 * w);
        }
        const bool partial = ntok < BS;
#pragma unroll
        for (int w = 0; w < CV / 8; ++w) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t sel = (uint32_t)k | ((uint32_t)k << 4) | ((uint32_t)(4 + k) << 8) | ((uint32_t)(4 + k) << 12);
            const uint32_t pAB = prmt(ra[w], rb[w], sel), pCD = prmt(rc[w], rd[w], sel);
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              uint32_t b0 = dq2(lop_nib(pAB >> (4 * e)), sA, mA);
              uint32_t b1 = dq2(lop_nib(pCD >> (4 * e)), sB, mB);
              if (partial) {
                b0 = b0 & ((t0 < ntok ? 0x0000ffffu : 0u) | (t0 + 1 < ntok ? 0xffff0000u : 0u));
                b1 = b1 & ((t0 + 8 < ntok ? 0x0000ffffu : 0u) | (t0 + 9 < ntok ? 0xffff0000u : 0u));
              }
              mma_f16(o[8 * w + 2 * k + e], pa, b0, b1);
              mma_f16(o[8 * w + 2 * k + e], pl, b0, b1);
            }
          }
        }
      }
    }

    if (flags & F_LAST) {
      float L0 = l0 + __shfl_xor_sync(FULL_MASK, l0, 1);
      L0 += __shfl_xor_sync(FULL_MASK, L0, 2);
      float L1 = l1 + __shfl_xor_sync(FULL_MASK, l1, 1);
      L1 += __shfl_xor_sync(FULL_MASK, L1, 2);
      const bool whole = flags & F_WHOLE;
      const float i0 = whole ? (L0 > 0.f ? 1.f / L0 : 0.f) : 1.f, i1 = whole ? (L1 > 0.f ? 1.f / L1 : 0.f) : 1.f;
      // Column n-slot 2*tig + e of n-tile nt holds channel (2*tig+e)*CV + 8*(nt/8) + channel_of(nt%8).
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        float r0v[CV], r1v[CV];
#pragma unroll
        for (int c = 0; c < CV; ++c) {
          const int nt = 8 * (c >> 3) + nibble_of(c & 7);
          r0v[c] = o[nt][e] * i0;
          r1v[c] = o[nt][2 + e] * i1;
        }
        const int c0 = (2 * tig + e) * CV;
        if (whole) {
          const size_t row0 = (size_t)s * a.n_h + (size_t)g * a.G + hl0;
          if (a.out_f32) {
            float* out0 = reinterpret_cast<float*>(a.out) + row0 * D + c0;
#pragma unroll
            for (int c = 0; c < CV; c += 4) {
              if (v0) *reinterpret_cast<float4*>(out0 + c) = make_float4(r0v[c], r0v[c + 1], r0v[c + 2], r0v[c + 3]);
              if (v1) *reinterpret_cast<float4*>(out0 + 8 * D + c) = make_float4(r1v[c], r1v[c + 1], r1v[c + 2], r1v[c + 3]);
            }
          } else {
            uint32_t* out0 = reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + row0 * D + c0);
#pragma unroll
            for (int c = 0; c < CV; c += 8) {
              if (v0)
                *reinterpret_cast<uint4*>(out0 + c / 2) =
                    make_uint4(pack_bf16(r0v[c], r0v[c + 1]), pack_bf16(r0v[c + 2], r0v[c + 3]),
                               pack_bf16(r0v[c + 4], r0v[c + 5]), pack_bf16(r0v[c + 6], r0v[c + 7]));
              if (v1)
                *reinterpret_cast<uint4*>(out0 + 4 * D + c / 2) =
                    make_uint4(pack_bf16(r1v[c], r1v[c + 1]), pack_bf16(r1v[c + 2], r1v[c + 3]),
                               pack_bf16(r1v[c + 4], r1v[c + 5]), pack_bf16(r1v[c + 6], r1v[c + 7]));
            }
          }
        } else {
          const long long part = (long long)s * a.n_kv + g + p;
          float* wo = a.ws_o + (size_t)part * a.G * D + c0;
#pragma unroll
          for (int c = 0; c < CV; c += 4) {
            if (v0) *reinterpret_cast<float4*>(wo + (size_t)hl0 * D + c) = make_float4(r0v[c], r0v[c + 1], r0v[c + 2], r0v[c + 3]);
            if (v1) *reinterpret_cast<float4*>(wo + (size_t)hl1 * D + c) = make_float4(r1v[c], r1v[c + 1], r1v[c + 2], r1v[c + 3]);
          }
        }
      }
      if (!whole && tig == 0) {
        const long long part = (long long)s * a.n_kv + g + p;
        if (v0) *reinterpret_cast<float2*>(a.ws_ml + ((size_t)part * a.G + hl0) * 2) = make_float2(m0, L0);
        if (v1) *reinterpret_cast<float2*>(a.ws_ml + ((size_t)part * a.G + hl1) * 2) = make_float2(m1, L1);
      }
    }

    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[slot]);
    if (warp == 0 && j + S < len) issue(j + S);
  }

  if (abort_flag && threadIdx.x == 0) {
    const int issued = len < consumed + S ? len : consumed + S;
    for (int j = consumed; j < issued; ++j)
      if (!mbar_wait(&full[j % S], (j / S) & 1)) break;
  }
}

// ---------------------------------------------------------------------------------------------
struct Int4Variant {
  const void* fn;
  int stages;
  size_t smem;
  int warps;
  int P;
};

template <int D, int BS, int MT>
static Int4Variant make_int4_variant() {
  Int4Variant v;
  v.fn = (const void*)decode_int4_kernel<D, BS, MT>;
  const int stage = Int4Tile<D, BS>::STAGE;
  v.stages = ring_stages(stage, "PKV_STAGES_INT4");
  v.smem = int4_smem_bytes<D, BS>(v.stages);
  v.warps = MT;
  v.P = 0;
  return v;
}

static Int4Variant* lookup_int4(int D, int BS, int MT) {
  static std::mutex mu;
  static Int4Variant table[2][3][3];
  static bool ready[2][3][3] = {};
  const int di = D == 128 ? 1 : 0, bi = BS == 16 ? 0 : (BS == 32 ? 1 : 2), mi = MT == 1 ? 0 : (MT == 2 ? 1 : 2);
  std::lock_guard<std::mutex> lock(mu);
  Int4Variant& v = table[di][bi][mi];
  if (!ready[di][bi][mi]) {
#define PKV_V(d, b, m) \
  if (D == d && BS == b && MT == m) v = make_int4_variant<d, b, m>();
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

int int4_pieces(int D, int BS, int G) {
  Int4Variant* v = lookup_int4(D, BS, mt_for_group(G));
  return v ? v->P : 0;
}

}  // namespace pkv

using namespace pkv;

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static bool valid_shape(int n_h, int n_kv, int head_dim, int block_size) {
  if (head_dim != 64 && head_dim != 128) return false;
  if (block_size != 16 && block_size != 32 && block_size != 64) return false;
  if (n_kv <= 0 || n_h <= 0 || n_h % n_kv) return false;
  return n_h / n_kv <= 64;
}

extern "C" pkv_status pkv_kv_quant_append_int4(const void* k, const void* v, const int64_t* slot_mapping,
                                               const int32_t* tail_seq, int n_tok, uint8_t* k_codes, void* k_meta,
                                               uint8_t* v_codes, void* v_meta, void* k_tail, int tail_rows,
                                               int num_blocks, int block_size, int n_kv, int head_dim,
                                               int32_t* err_flag, void* stream) {
  if (n_tok < 0 || num_blocks < 0 || n_kv <= 0 || tail_rows < 0) return PKV_EINVAL;
  if (head_dim != 64 && head_dim != 128) return PKV_EINVAL;
  if (block_size != 16 && block_size != 32 && block_size != 64) return PKV_EINVAL;
  if (n_tok == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !tail_seq || !k_codes || !k_meta || !v_codes || !v_meta || !k_tail)
    return PKV_EINVAL;
  if (!al16(k) || !al16(v) || !al16(k_codes) || !al16(v_codes) || !al16(k_meta) || !al16(v_meta) || !al16(k_tail))
    return PKV_EINVAL;
  QuantAppendArgs a;
  a.k = static_cast<const __nv_bfloat16*>(k);
  a.v = static_cast<const __nv_bfloat16*>(v);
  a.slots = slot_mapping;
  a.tail_seq = tail_seq;
  a.n_tok = n_tok;
  a.n_kv = n_kv;
  a.block_size = block_size;
  a.tail_rows = tail_rows;
  a.n_slots = (long long)num_blocks * block_size;
  a.k_codes = k_codes;
  a.k_meta = static_cast<__half*>(k_meta);
  a.v_codes = v_codes;
  a.v_meta = static_cast<__half*>(v_meta);
  a.k_tail = static_cast<__nv_bfloat16*>(k_tail);
  a.err = err_flag;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long warps = (long long)n_tok * n_kv;
  const unsigned g1 = (unsigned)((warps * 32 + 255) / 256);
  const long long vecs = warps * (head_dim / 8);
  const unsigned g2 = (unsigned)((vecs + 255) / 256);
  if (head_dim == 128) {
    quant_append_kernel<128><<<g1, 256, 0, st>>>(a);
    tail_write_kernel<128><<<g2, 256, 0, st>>>(a);
  } else {
    quant_append_kernel<64><<<g1, 256, 0, st>>>(a);
    tail_write_kernel<64><<<g2, 256, 0, st>>>(a);
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}

extern "C" pkv_status pkv_paged_decode_attn_int4(const void* q, const uint8_t* k_codes, const void* k_meta,
                                                 const uint8_t* v_codes, const void* v_meta, const void* k_tail,
                                                 const int32_t* block_tables, int max_blocks,
                                                 const int32_t* context_lens, float scale, int batch, int n_h,
                                                 int n_kv, int head_dim, int block_size, int num_blocks, void* out,
                                                 int out_dtype, void* workspace, size_t workspace_bytes,
                                                 int32_t* err_flag, void* stream) {
  if (batch < 0 || !valid_shape(n_h, n_kv, head_dim, block_size) || max_blocks < 0 || num_blocks < 0)
    return PKV_EINVAL;
  if (out_dtype != PKV_OUT_BF16 && out_dtype != PKV_OUT_F32) return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  if (!q || !k_codes || !k_meta || !v_codes || !v_meta || !k_tail || !block_tables || !context_lens || !out ||
      !workspace)
    return PKV_EINVAL;
  if (!al16(q) || !al16(k_codes) || !al16(v_codes) || !al16(k_meta) || !al16(v_meta) || !al16(k_tail) ||
      !al16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_EINVAL;
  if ((long long)max_blocks * block_size > 0x7fffffffLL) return PKV_ERANGE;
  const int G = n_h / n_kv;
  Int4Variant* vv = lookup_int4(head_dim, block_size, mt_for_group(G));
  if (!vv) {
    record_cuda_error(cudaGetLastError());
    return PKV_ECUDA;
  }
  const WorkspaceLayout wl = workspace_layout(batch, n_kv, G, head_dim, vv->P);
  if (workspace_bytes < wl.total) return PKV_ENOSPC;
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
  a.stages = vv->stages;
  a.k_codes = k_codes;
  a.v_codes = v_codes;
  a.k_meta = static_cast<const __half*>(k_meta);
  a.v_meta = static_cast<const __half*>(v_meta);
  a.k_tail = static_cast<const __nv_bfloat16*>(k_tail);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = a.inline_plan ? cudaSuccess
                                : launch_plan(context_lens, batch, max_blocks * block_size, block_size, a, vv->P, st);
  if (e == cudaSuccess) {
    void* kargs[] = {&a};
    e = launch_pdl(vv->fn, dim3(vv->P), dim3(vv->warps * 32), vv->smem, st, kargs);
  }
  if (e == cudaSuccess) e = launch_reduce(head_dim, a, vv->P, st);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}
