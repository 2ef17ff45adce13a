// INT4 paged KV cache: quantize-on-append, and decode attention over the exact codes with
// the scales folded into the other operands.  Format and exact quantizer op sequence are
// documented in pkv.h.
#include <cmath>
#include <mutex>

#include "decode_common.cuh"
#include "nvtx_range.h"

namespace pkv {

// nibble index (0..7) inside a 32-bit word of the code row that holds channel c' (0..7)
__host__ __device__ constexpr int nibble_of(int c) { return (c & 1) ? 4 + (c >> 1) : (c >> 1); }
// channel offset held by nibble n
__host__ __device__ constexpr int channel_of(int n) { return n < 4 ? 2 * n : 2 * (n - 4) + 1; }

struct GroupQuant {
  float s, m;           // fp16 scale / min, widened
  float r;              // 1 / s rounded to nearest (0 when s is 0)
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
  q.r = q.s == 0.f ? 0.f : __frcp_rn(q.s);
  return q;
}
// Step (4): code of one value, rint((x - m) / s) with the quotient rounded to nearest,
// clamped to [0, 15].  Where the clamp does not decide the code, |quotient| <= 16, and the
// product with the rounded reciprocal is then within 3e-6 of the rounded quotient (each is
// within 2^-23 relative of the exact one); so when the product lies more than 1e-5 from
// every half-integer both round to the same integer, and only near a tie is the division
// itself taken.  NaN and infinite inputs give the same codes either way.
__device__ __forceinline__ uint32_t quant_code(float x, const GroupQuant& q) {
  if (q.s == 0.f) return 0u;
  const float d = __fsub_rn(x, q.m);
  const float t = __fmul_rn(d, q.r);
  float c = rintf(t);
  if (fabsf(fabsf(t - c) - 0.5f) < 1e-5f) c = rintf(__fdiv_rn(d, q.s));
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
  uint8_t* cache;                 // [num_blocks][n_kv][rec_bytes] records
  size_t rec_bytes;
  __nv_bfloat16* k_tail;
  int32_t* err;
};

// Phase 1: D / 32 warps per (token, kv head).  The first quantizes V per token; when the
// token fills the last row of its block, each of them quantizes 32 of that block's K
// channels (per channel), taking rows appended earlier in this call from `k` and older rows
// from the tail.
template <int D>
constexpr int kKWarps = D / 32;                 // warps per (token, kv head)
template <int D, int BS>
__global__ void __launch_bounds__(256) quant_append_kernel(const QuantAppendArgs a) {
  grid_dep_launch();                            // the tail update may launch; it waits for this grid
  constexpr int CPL = D / 32;                   // V channels per lane
  constexpr int LPW = 8 / CPL;                  // lanes per 32-bit code word
  constexpr int KQ = kKWarps<D>;
  const int lane = threadIdx.x & 31;
  const long long wall = (blockIdx.x * (long long)blockDim.x + threadIdx.x) >> 5;
  const long long wid = wall / KQ;
  const int kq = (int)(wall - wid * KQ);        // this warp's 32 K channels: [32 kq, 32 kq + 32)
  if (wid >= (long long)a.n_tok * a.n_kv) return;
  const int i = (int)(wid / a.n_kv), g = (int)(wid % a.n_kv);
  const long long slot = a.slots[i];
  if (slot < 0) return;
  const int seq = a.tail_seq[i];
  if (slot >= a.n_slots || (unsigned)seq >= (unsigned)a.tail_rows) {
    if (lane == 0 && g == 0 && kq == 0) set_err(a.err, PKV_DEV_BAD_SLOT);
    return;
  }
  const long long blk = slot / BS;
  const int row = (int)(slot - blk * BS);
  const size_t tile = (size_t)blk * a.n_kv + g;           // (block, kv head)
  uint8_t* rec = a.cache + tile * a.rec_bytes;            // K codes, V codes, K meta, V meta

  // ---- V: per token ----
  if (kq == 0) {
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
    uint32_t* dst = reinterpret_cast<uint32_t*>(rec + (size_t)(BS + row) * (D / 2));
    if (lane % LPW == 0) dst[lane / LPW] = word;
    if (lane == 0) {
      __half2 meta = __halves2half2(q.s16, q.m16);
      reinterpret_cast<__half2*>(rec + (size_t)BS * D + 4 * D)[row] = meta;
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
  __half* kmeta = reinterpret_cast<__half*>(rec + (size_t)BS * D);
  uint32_t* kcodes = reinterpret_cast<uint32_t*>(rec);
  // Lane (octet, row group): channels [8 octet, 8 octet + 8) of this warp's 32 -- one code
  // word per row -- of the rows r0 + rg + RG k of each chunk of KR rows, loaded as 16-byte
  // vectors, every load of a chunk issued before any is used.  The channel range comes from
  // a min / max over the lane's rows and then across the row groups; a block of KR rows
  // stays in registers from the range pass to the code pass.
  constexpr int OCT = 4;                                     // channel octets per warp
  constexpr int RG = 32 / OCT;                               // row groups
  constexpr int KR = 16;                                     // rows per chunk
  constexpr int RPL = KR / RG;                               // rows per lane and chunk
  const int oct = kq * OCT + lane % OCT, rg = lane / OCT;     // oct: octet within the row
  auto row_ptr = [&](int r) -> const __nv_bfloat16* {
    return r >= first_call_row ? krow_call + (size_t)(i - (BS - 1 - r)) * a.n_kv * D : krow_tail + (size_t)r * D;
  };
  float x[RPL][8];
  auto load_chunk = [&](int r0) {
    uint4 v[RPL];
#pragma unroll
    for (int k = 0; k < RPL; ++k) v[k] = *reinterpret_cast<const uint4*>(row_ptr(r0 + rg + RG * k) + 8 * oct);
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        x[k][2 * e] = bf16_lo(w[e]);
        x[k][2 * e + 1] = bf16_hi(w[e]);
      }
    }
  };
  float lo[8], hi[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    lo[c] = INFINITY;
    hi[c] = -INFINITY;
  }
#pragma unroll 1
  for (int r0 = 0; r0 < BS; r0 += KR) {
    load_chunk(r0);
#pragma unroll
    for (int k = 0; k < RPL; ++k)
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        lo[c] = fminf(lo[c], x[k][c]);
        hi[c] = fmaxf(hi[c], x[k][c]);
      }
  }
  GroupQuant q[8];
#pragma unroll
  for (int c = 0; c < 8; ++c) {
#pragma unroll
    for (int o = OCT; o < 32; o <<= 1) {                     // across the row groups
      lo[c] = fminf(lo[c], __shfl_xor_sync(FULL_MASK, lo[c], o));
      hi[c] = fmaxf(hi[c], __shfl_xor_sync(FULL_MASK, hi[c], o));
    }
    q[c] = group_params(lo[c], hi[c]);
  }
  if (rg == 0) {
    uint32_t sv[4], mv[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half2 s2 = __halves2half2(q[2 * e].s16, q[2 * e + 1].s16);
      const __half2 m2 = __halves2half2(q[2 * e].m16, q[2 * e + 1].m16);
      sv[e] = *reinterpret_cast<const uint32_t*>(&s2);
      mv[e] = *reinterpret_cast<const uint32_t*>(&m2);
    }
    *reinterpret_cast<uint4*>(kmeta + 8 * oct) = make_uint4(sv[0], sv[1], sv[2], sv[3]);
    *reinterpret_cast<uint4*>(kmeta + D + 8 * oct) = make_uint4(mv[0], mv[1], mv[2], mv[3]);
  }
#pragma unroll 1
  for (int r0 = 0; r0 < BS; r0 += KR) {
    if (BS > KR) load_chunk(r0);                             // else the rows are still in registers
#pragma unroll
    for (int k = 0; k < RPL; ++k) {
      uint32_t word = 0;
#pragma unroll
      for (int c = 0; c < 8; ++c) word |= quant_code(x[k][c], q[c]) << (4 * nibble_of(c));
      kcodes[(size_t)(r0 + rg + RG * k) * (D / 8) + oct] = word;
    }
  }
}

// Phase 2: K rows of blocks that stay unfinished after this call go to the tail.
template <int D>
__global__ void __launch_bounds__(256) tail_write_kernel(const QuantAppendArgs a) {
  // The tail rows of a block this call completes are read by phase 1: wait for it before
  // writing any.  The attention's setup may overlap this kernel.
  grid_dep_wait();
  grid_dep_launch();
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
// Same partition, producer and token-major tiles as the bf16 kernel.  A stage holds one
// (block, kv head) record -- K codes [BS][D/2], V codes [BS][D/2], K meta [2][D] fp16,
// V meta [BS][2] fp16 -- moved by one 1-D bulk copy, or with TB = 2 two records of
// consecutive blocks of one segment.  A sequence's unfinished last block has no K codes:
// its K rows are read from the bf16 tail straight from L2 (the producer prefetches them
// when it enters the segment), so the ring holds no tail space.
//
// No value is dequantized: the scales are folded into the other operand, so the result is
// the attention over the exact x^ = code * s + min up to fp32 accumulation.
//
// S^T = K^ Q^T, fp16 mma.  K^[t][c] = code * s_c + m_c with a per-channel (s, m) per
// block, so  q . k^_t = sum_c (16 + code_tc) (q_c s_c) + sum_c q_c (m_c - 16 s_c).
// The A operand is 16 + code, exact in fp16, made from a nibble pair by one shift and one
// mask-and-or (the code lands in mantissa bits 6..9 under the exponent of 16).  The B
// operand is q * s, carried as an fp16 high part and the exact residual (q is bf16 and s
// fp16, so their product has at most 19 significant bits: high + low holds it exactly).
// The second sum, a constant of the block per head, is one more mma chain with the min
// row and the scale row of the block as A rows 0 and 1 and q as B; it initialises the
// score accumulators.  For groups of up to 4 heads the 8-head n-tile carries the high
// part in columns 0-3 and the low part in columns 4-7, so one mma takes both and one
// shuffle adds the halves.  The channel order inside a k-step is permuted so each thread's
// A-fragment rows come from one 16-byte load of a token row: thread t of a quad owns
// channels [t*D/4, (t+1)*D/4); k-step ks takes word ks/2 and, inside it, channel pairs
// (0,1),(2,3) or (4,5),(6,7); Q^T uses the same order.
//
// O^T = V^T P^T, bf16 mma.  V^[t][c] = code * s_t + m_t with a per-token (s, m), so
//   sum_t p_t v^_tc = sum_t (code_tc - 8) (p_t s_t) + sum_t p_t (m_t + 8 s_t).
// The A operand is code - 8, exact in bf16 (mask-and-or into 128 + code, minus 136),
// centred so the accumulated terms have both signs; the B operand is p * s as a bf16 high
// + low pair; the second sum is a per-head fp32 scalar that each thread accumulates over
// its tokens and that is added to every channel at the end.  Thread g of the eight row
// groups owns channels [g*D/8, (g+1)*D/8); a byte of a V code word, permuted together from
// two token rows, gives a pair of two tokens of one channel (the even nibble for fragment
// row g, the odd one for row g+8).  For groups of up to 4 heads the P^T columns 4-7 carry
// the low part, as for the scores.
template <int D, int BS>
struct Int4Tile {
  static constexpr int KC = 0;                              // K codes [BS][D/2]
  static constexpr int VC = BS * D / 2;                     // V codes [BS][D/2]
  static constexpr int KM = BS * D;                         // K meta [2][D] fp16
  static constexpr int VM = BS * D + 4 * D;                 // V meta [BS][2] fp16
  static constexpr int REC = BS * D + 4 * D + 4 * BS;                 // one cache record
  static constexpr int STAGE = (REC + 127) / 128 * 128;
};

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ uint32_t and_or(uint32_t x, uint32_t mask, uint32_t bits) {   // (x & mask) | bits
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xea;" : "=r"(d) : "r"(x), "r"(mask), "r"(bits));
  return d;
}
__device__ __forceinline__ uint32_t xor_and(uint32_t x, uint32_t y, uint32_t mask) {     // (x ^ y) & mask
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0x28;" : "=r"(d) : "r"(x), "r"(y), "r"(mask));
  return d;
}
// fp16 pair (16 + code of nibble j, 16 + code of nibble j + 4) of a K code word: the
// nibbles sit at bits 4j and 16 + 4j and move to mantissa bits 6..9 of each half.
__device__ __forceinline__ uint32_t k_codes16(uint32_t w, int j) {
  const uint32_t x = j == 0 ? w << 6 : (j == 1 ? w << 2 : (j == 2 ? w >> 2 : w >> 6));
  return and_or(x, 0x03c003c0u, 0x4c004c00u);
}
// bf16 pair (code - 8) of the nibbles at bits 0..3 and 16..19: 128 + code by a
// mask-and-or (mantissa bits 0..3 under the exponent of 128), then minus 136, exactly.
__device__ __forceinline__ uint32_t v_codes8(uint32_t x) {
  const uint32_t c = and_or(x, 0x000f000fu, 0x43004300u);
  const __nv_bfloat162 r = __hsub2(*reinterpret_cast<const __nv_bfloat162*>(&c),
                                   __bfloat162bfloat162(__ushort_as_bfloat16(0x4308)));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hmul2_u(uint32_t a, uint32_t b) {
  const __half2 r = __hmul2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t hfma2_u(uint32_t a, uint32_t b, uint32_t c) {
  const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&a), *reinterpret_cast<const __half2*>(&b),
                            *reinterpret_cast<const __half2*>(&c));
  return *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ uint32_t bf2_to_h2(uint32_t w) { return pack_f16(bf16_lo(w), bf16_hi(w)); }
__device__ __forceinline__ float h_lo(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w & 0xffffu))); }
__device__ __forceinline__ float h_hi(uint32_t w) { return __half2float(__ushort_as_half((unsigned short)(w >> 16))); }

// TB cache records (blocks) per ring stage; a zero line after the barriers feeds the A rows
// of the bias product that carry nothing.
template <int D, int BS, int TB>
__host__ __device__ constexpr size_t int4_smem_bytes(int stages) {
  return 128 + (size_t)stages * (TB * Int4Tile<D, BS>::STAGE + 16 + 16) + 2 * D;
}

// softmax_tile plus the per-head correction sums of the V fold, rescaled with l and O when
// the running offset rises.
template <int TT, int NH, int MD>
__device__ __forceinline__ void softmax_tile_c(float (&sc)[TT][NH][4], float (&m)[NH][2], float (&l)[NH][2],
                                               float (&c)[NH][2], float (&o)[MD][NH][4], int gid, int ntok,
                                               int lead, float scale_log2) {
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
        c[nh][e] *= al[e];
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
// TB = 2: a stage holds two consecutive blocks of one segment when the piece has them
// (32 token rows per pass at block size 16: the per-stage loop, barrier, producer and
// softmax work is shared by twice the tokens).  COMB: groups of up to 4 heads, high and
// low parts of the folded operands in the two halves of one 8-head n-tile.
template <int D, int BS, int NH, int MT, int TB, bool COMB>
__global__ void __launch_bounds__(MT * 32, TB == 2 || (BS == 64 && MT == 1) ? 12 : (BS == 16 && MT == 1 && NH == 1 ? 16 : 0))
    decode_int4_kernel(const DecodeArgs a) {
  using T = Int4Tile<D, BS>;
  constexpr int TPB = BS / 16;      // 16-token tiles per block
  constexpr int TT = TB * TPB;      // 16-token tiles per stage
  constexpr int SST = TB * T::STAGE;
  constexpr int KS = D / 16;        // k-steps of K Q^T
  constexpr int MD = D / 16;        // 16-channel m-tiles of O^T
  constexpr int HW = 8 * NH;        // heads per warp
  constexpr int KW = D / 32;        // K code words per thread per token row
  constexpr int CB = D / 4;         // K channels per thread (k-slots of the QK fragments)
  constexpr int CV = D / 8;         // V channels per thread (rows of the V^T fragments)
  constexpr int VW = CV / 8;        // V code words per thread per token row
  extern __shared__ uint8_t smem_raw[];
  // aligned by an offset from the array itself, so every access stays a shared-memory one
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  const int S = a.stages;
  int4* meta = reinterpret_cast<int4*>(smem + (size_t)S * SST);
  uint64_t* full = reinterpret_cast<uint64_t*>(meta + S);
  uint64_t* empty = full + S;
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tig = lane & 3, gid = lane >> 2;

  uint32_t* zline = reinterpret_cast<uint32_t*>(empty + S);     // 2 * D zero bytes
  for (int i = threadIdx.x; i < D / 2; i += MT * 32) zline[i] = 0u;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int i = 0; i < S; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], MT);
    }
    fence_barrier_init();
  }
  __syncthreads();
  if (!a.inline_plan) grid_dep_wait();   // the plan kernel's cum / ctx_eff / cursors
  grid_dep_launch();

  Cursor cur;
  PieceInfo pi;
  piece_setup(a, blockIdx.x, gridDim.x, warp == 0, cur, pi);
  const int P = pi.P, p = blockIdx.x;
  const long long pstart = pi.pstart, pend = pi.pend;
  const int len = p < P ? (int)(pend - pstart) : 0;
  // A CTA without work still waits for the kernel before it (in inline-plan mode its
  // wait comes below), so no launch after this grid on the stream can pass the append.
  if (len <= 0) {
    if (a.inline_plan) grid_dep_wait();
    return;
  }
  // The setup above reads only this call's inputs; the cache and the K tail may still be
  // being written by the kernel before this one on the stream (the quantize-on-append),
  // so every thread waits for it here, with the piece's first block-table line on its way.
  if (warp == 0 && lane == 0) prefetch_l2(a.bt + (size_t)cur.s * a.max_blocks + cur.b0 + cur.blk);
  if (a.inline_plan) grid_dep_wait();

  int w_seq = -1, w_base = 0, w_phys = -1, n_seq = -1, n_base = 0, n_phys = -1;
  const uint64_t pol = policy_evict_first();
  // ring position of the next issue / the next stage consumed (slot, and the parity of the
  // pass over the ring), advanced in order instead of dividing by the stage count
  int p_slot = 0, c_slot = 0;
  uint32_t p_phase = 0, c_phase = 0;
  int pj = 0;                       // next block of the piece to issue (producer warp)
  int issued = 0;                   // stages issued (producer warp)

  const uint32_t ring_sa = smem_u32(smem);                   // ring, then meta[S], then full[S]
  // constants of the segment the producer is in, set when it enters one: its last block,
  // and pack_rows(rows of the last block, rows of block 0 before the window, F_WHOLE)
  int seg_last = 0, seg_rows = 0;

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
    const bool first = pj == 0 || cur.blk == 0;
    if (first) {
      seg_last = cur.nb - 1;
      seg_rows = pack_rows(cur.ctx - (cur.b0 + seg_last) * BS, window_lead(cur.ctx, a.window, BS),
                           cur.seg_start >= pstart && cur.seg_start + cur.nb <= pend ? F_WHOLE : 0);
      const char* qp = reinterpret_cast<const char*>(a.q) + ((size_t)cur.s * a.n_h + (size_t)cur.g * a.G) * D * 2;
      for (int off = lane * 128; off < a.G * D * 2; off += 32 * 128) prefetch_l2(qp + off);
      if (cur.ctx % BS) {                                      // warm L2 with the bf16 tail early
        const char* tail = reinterpret_cast<const char*>(a.k_tail + ((size_t)cur.s * a.n_kv + cur.g) * BS * D);
        for (int off = lane * 128; off < 2 * BS * D; off += 32 * 128) prefetch_l2(tail + off);
      }
    }
    // A single consumer warp is this warp: the slot refilled here is the one it released
    // just before (after __syncwarp, every value read from it already used), so only the
    // order of its generic-proxy reads before the async-proxy writes is needed.  Several
    // consumer warps release the slot through the empty barrier.
    bool ok_wait = true;
    if (MT > 1 && issued >= S) {
      if (lane == 0) ok_wait = mbar_wait(&empty[slot], ph ^ 1u);   // released in the previous pass
      ok_wait = __shfl_sync(FULL_MASK, ok_wait, 0);
    }
    const int nblk = pair ? 2 : 1;
    const bool last = cur.blk + nblk - 1 == seg_last;
    const int ntok = (nblk - 1) * BS + (last ? (seg_rows & 255) : BS);   // rows of the stage
    const bool ok = (unsigned)phys < (unsigned)a.num_blocks && (!pair || (unsigned)phys1 < (unsigned)a.num_blocks);
    const bool go = ok && ok_wait, end = pj + nblk >= len;
    const int flags = (seg_rows >> 8 & F_WHOLE) | (ok ? F_VALID : 0) | (first ? F_FIRST : 0) |
                      (last || end ? F_LAST : 0) | (pair ? F_PAIR : 0) | (end ? F_END : 0);
    if (lane == 0) {
      if (!ok_wait) {
        set_err(a.err, PKV_DEV_TIMEOUT);
        abort_flag = 1;
      }
      if (!ok) set_err(a.err, PKV_DEV_BAD_BLOCK);
      meta[slot] = make_int4(cur.s, cur.g, cur.blk, pack_rows(ntok, cur.blk == 0 ? seg_rows >> 16 : 0, flags));
      if (go) {
        // whole records, also for the unfinished block (its K codes are then unused)
        const uint32_t bar = ring_sa + S * (SST + 16) + 8u * (uint32_t)slot;
        const uint32_t dst = ring_sa + (uint32_t)slot * SST;
        mbar_arrive_expect_tx(&full[slot], nblk * T::REC);
        if (MT == 1 && issued >= S) fence_proxy_async_smem();
        bulk_g2s_u32(dst, a.cache + ((size_t)(unsigned)phys * (unsigned)a.n_kv + (unsigned)cur.g) * T::REC, T::REC,
                     bar, pol);
        if (pair)
          bulk_g2s_u32(dst + T::STAGE,
                       a.cache + ((size_t)(unsigned)phys1 * (unsigned)a.n_kv + (unsigned)cur.g) * T::REC, T::REC,
                       bar, pol);
      } else {
        mbar_arrive(&full[slot]);
      }
    }
    if (pair) ++cur.blk;                                       // the second block, same segment
    pj += nblk;
    ++issued;
    if (pj < len) cursor_next(cur, a);
  };

  // ---------------- consumer state (warp w: local heads [w*HW, (w+1)*HW)) ----------------
  // Token-major tiles as in the bf16 kernel.  qb: q in fp16 (exact for bf16 values in fp16
  // range) as QK B fragments in the permuted channel order; with COMB, column n holds head
  // n % 4 (columns 4-7 repeat 0-3 and carry the low parts of the folded products).
  uint32_t qb[KS][NH][2];
  float o[MD][NH][4];
  float m[NH][2], l[NH][2], cs[NH][2];        // running offset, sum, V-fold correction
  const int hw0 = warp * HW;
  const int cb = tig * CB;           // first K channel of this thread
  const int cv = gid * CV;           // first V channel of this thread
  // A rows of the bias product: row 0 the block's K min row, row 1 its K scale row, the
  // other rows read the zero line
  const int xrow = gid == 0 ? T::KM + 2 * D : (gid == 1 ? T::KM : -1);
  const uint32_t lo_lane = COMB && gid >= 4 ? 0xffffffffu : 0u;  // columns 4-7: low parts

  if (warp == 0)
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
    // ntok, lead: the stage's attended rows are [lead, ntok) of its TT * 16
    const int s = mt.x, g = mt.y, ntok = mt.w & 255, flags = (mt.w >> 8) & 255, lead = mt.w >> 16;
    const size_t qrow0 = (size_t)s * a.n_h + (size_t)g * a.G;

    if (flags & F_FIRST) {
#pragma unroll
      for (int nh = 0; nh < NH; ++nh) {
        const int hl = COMB ? (gid & 3) : hw0 + nh * 8 + gid;
        const uint32_t* qp = reinterpret_cast<const uint32_t*>(a.q) + (qrow0 + hl) * (D / 2);
        const bool ok = hl < a.G;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const int w = (cb >> 1) + 4 * (ks >> 1) + 2 * (ks & 1);   // channel pair cb + 2*pr
          qb[ks][nh][0] = ok ? bf2_to_h2(__ldg(qp + w)) : 0u;
          qb[ks][nh][1] = ok ? bf2_to_h2(__ldg(qp + w + 1)) : 0u;
        }
        m[nh][0] = m[nh][1] = -INFINITY;
        l[nh][0] = l[nh][1] = 0.f;
        cs[nh][0] = cs[nh][1] = 0.f;
#pragma unroll
        for (int md = 0; md < MD; ++md) o[md][nh][0] = o[md][nh][1] = o[md][nh][2] = o[md][nh][3] = 0.f;
      }
    }

    if (flags & F_VALID) {
      const uint8_t* stg = smem + (size_t)slot * SST;
      const int nblk = TB > 1 && (flags & F_PAIR) ? 2 : 1;      // records in the stage
      // the stage's last record is the sequence's unfinished block (K from the tail) when
      // its rows stop short of the block
      const int tail_rec = ntok < nblk * BS ? nblk - 1 : -1;   // (at most one record per stage)
      const bool masked = ntok < TT * 16 || lead > 0;
      // ---- S^T = K^ Q^T (fp16 in, fp32 accumulate; two accumulators per tile) ----
      float sc[TT][NH][4], sx[TT][NH][4];
#pragma unroll
      for (int t = 0; t < TT; ++t)
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int i = 0; i < 4; ++i) sc[t][nh][i] = sx[t][nh][i] = 0.f;
#pragma unroll
      for (int rec = 0; rec < TB; ++rec) {
        if (rec >= nblk) continue;
        const uint8_t* st = stg + rec * T::STAGE;
        if (rec != tail_rec) {
          uint32_t s2[CB / 2], x2[CB / 2];             // scale pairs of channels cb + 2k; bias A rows
          {
            const uint4* ks4 = reinterpret_cast<const uint4*>(st + T::KM + cb * 2);
            const uint4* xs4 = reinterpret_cast<const uint4*>(
                (xrow >= 0 ? st + xrow : reinterpret_cast<const uint8_t*>(zline)) + cb * 2);
#pragma unroll
            for (int k4 = 0; k4 < CB / 8; ++k4) {
              const uint4 a4 = ks4[k4], b4 = xs4[k4];
              s2[4 * k4] = a4.x; s2[4 * k4 + 1] = a4.y; s2[4 * k4 + 2] = a4.z; s2[4 * k4 + 3] = a4.w;
              x2[4 * k4] = b4.x; x2[4 * k4 + 1] = b4.y; x2[4 * k4 + 2] = b4.z; x2[4 * k4 + 3] = b4.w;
            }
          }
          // bias of each head column: sum_c q_c m_c - 16 sum_c q_c s_c (rows 0 and 1 of one
          // mma chain), the starting value of the block's score accumulators
#pragma unroll
          for (int nh = 0; nh < NH; ++nh) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              const int pr = 4 * (ks >> 1) + 2 * (ks & 1);
              const uint32_t xa[4] = {x2[pr], 0u, x2[pr + 1], 0u};
              mma_f16(d, xa, qb[ks][nh][0], qb[ks][nh][1]);
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const float bm = __shfl_sync(FULL_MASK, d[e], tig);
              const float bsq = __shfl_sync(FULL_MASK, d[e], 4 + tig);
              const float bias = (COMB && tig >= 2) ? 0.f : fmaf(-16.f, bsq, bm);
#pragma unroll
              for (int tt = 0; tt < TPB; ++tt) {
                sc[rec * TPB + tt][nh][e] = bias;
                sc[rec * TPB + tt][nh][2 + e] = bias;
              }
            }
          }
          uint32_t w0[TPB][KW], w1[TPB][KW];                       // code words of rows gid, gid+8
#pragma unroll
          for (int tt = 0; tt < TPB; ++tt) {
            const uint8_t* q0 = st + T::KC + (tt * 16 + gid) * (D / 2) + tig * (D / 8);
            const uint8_t* q1 = q0 + 8 * (D / 2);
            if constexpr (KW == 4) {
              const uint4 x = *reinterpret_cast<const uint4*>(q0), y = *reinterpret_cast<const uint4*>(q1);
              w0[tt][0] = x.x; w0[tt][1] = x.y; w0[tt][2] = x.z; w0[tt][3] = x.w;
              w1[tt][0] = y.x; w1[tt][1] = y.y; w1[tt][2] = y.z; w1[tt][3] = y.w;
            } else {
              const uint2 x = *reinterpret_cast<const uint2*>(q0), y = *reinterpret_cast<const uint2*>(q1);
              w0[tt][0] = x.x; w0[tt][1] = x.y;
              w1[tt][0] = y.x; w1[tt][1] = y.y;
            }
          }
#pragma unroll
          for (int ks = 0; ks < KS; ++ks) {
            const int w = ks >> 1, j0 = 2 * (ks & 1), pr = 4 * w + j0;
            // B: q * s, high part and exact low part (COMB: the low part in columns 4-7)
            uint32_t bh[NH][2], bl[NH][2];
#pragma unroll
            for (int nh = 0; nh < NH; ++nh)
#pragma unroll
              for (int j = 0; j < 2; ++j) {
                const uint32_t hi = hmul2_u(qb[ks][nh][j], s2[pr + j]);
                if (COMB) {
                  bh[nh][j] = hfma2_u(qb[ks][nh][j], s2[pr + j], xor_and(hi, 0x80008000u, lo_lane));
                } else {
                  bh[nh][j] = hi;
                  bl[nh][j] = hfma2_u(qb[ks][nh][j], s2[pr + j], hi ^ 0x80008000u);
                }
              }
#pragma unroll
            for (int tt = 0; tt < TPB; ++tt) {
              const int t = rec * TPB + tt;
              uint32_t ka[4];
              ka[0] = k_codes16(w0[tt][w], j0);
              ka[1] = k_codes16(w1[tt][w], j0);
              ka[2] = k_codes16(w0[tt][w], j0 + 1);
              ka[3] = k_codes16(w1[tt][w], j0 + 1);
#pragma unroll
              for (int nh = 0; nh < NH; ++nh) {
                if (COMB) {
                  if (ks & 1) mma_f16(sx[t][nh], ka, bh[nh][0], bh[nh][1]);
                  else mma_f16(sc[t][nh], ka, bh[nh][0], bh[nh][1]);
                } else {
                  mma_f16(sc[t][nh], ka, bh[nh][0], bh[nh][1]);
                  mma_f16(sx[t][nh], ka, bl[nh][0], bl[nh][1]);
                }
              }
            }
          }
        } else {
          // unfinished block: K rows from the bf16 tail in global memory (prefetched to L2),
          // converted to fp16 (exact in range), against q itself
          const uint4* tl = reinterpret_cast<const uint4*>(a.k_tail + ((size_t)s * a.n_kv + g) * BS * D);
#pragma unroll
          for (int tt = 0; tt < TPB; ++tt) {
            const int t = rec * TPB + tt;
            uint32_t w0[CB / 2], w1[CB / 2];                      // bf16 pairs of channels cb + 2k
            const uint4* q0 = tl + ((size_t)(tt * 16 + gid) * D + cb) / 8;
            const uint4* q1 = q0 + D;                             // 8 rows further (D / 8 uint4 per row)
#pragma unroll
            for (int k4 = 0; k4 < CB / 8; ++k4) {
              const uint4 x = __ldg(q0 + k4), y = __ldg(q1 + k4);
              w0[4 * k4] = x.x; w0[4 * k4 + 1] = x.y; w0[4 * k4 + 2] = x.z; w0[4 * k4 + 3] = x.w;
              w1[4 * k4] = y.x; w1[4 * k4 + 1] = y.y; w1[4 * k4 + 2] = y.z; w1[4 * k4 + 3] = y.w;
            }
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
              const int pr = 4 * (ks >> 1) + 2 * (ks & 1);
              uint32_t ka[4];
              ka[0] = bf2_to_h2(w0[pr]);
              ka[1] = bf2_to_h2(w1[pr]);
              ka[2] = bf2_to_h2(w0[pr + 1]);
              ka[3] = bf2_to_h2(w1[pr + 1]);
#pragma unroll
              for (int nh = 0; nh < NH; ++nh) {
                if (ks & 1) mma_f16(sx[t][nh], ka, qb[ks][nh][0], qb[ks][nh][1]);
                else mma_f16(sc[t][nh], ka, qb[ks][nh][0], qb[ks][nh][1]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const bool comb_tile = COMB && t / TPB < nblk && t / TPB != tail_rec;
#pragma unroll
        for (int nh = 0; nh < NH; ++nh)
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            float x = sc[t][nh][i] + sx[t][nh][i];
            // COMB: the high-part sums (columns 0-3) and the low-part sums (4-7) of the same
            // heads, added in both halves (the tail block's two halves already hold the score)
            if (COMB) {
              const float y = __shfl_xor_sync(FULL_MASK, x, 2);
              if (comb_tile) x += y;
            }
            sc[t][nh][i] = x;
          }
      }
      softmax_tile_c<TT, NH, MD>(sc, m, l, cs, o, gid, ntok, lead, a.scale_log2);
      // ---- O^T += V^T P'^T (bf16, P' = p * s_t as high + low) ----
#pragma unroll
      for (int t = 0; t < TT; ++t) {
        const int rec = t / TPB, r0 = (t % TPB) * 16;             // record, first row in it
        if (rec >= nblk) continue;
        const uint8_t* st = stg + rec * T::STAGE;
        const uint32_t* vm = reinterpret_cast<const uint32_t*>(st + T::VM);
        // (s, m) of this thread's token rows gid and gid + 8; rows outside [lead, ntok) get
        // 0 and 0 (their p is 0 and their metadata may never have been written)
        uint32_t u0 = vm[r0 + gid], u1 = vm[r0 + gid + 8];
        if (masked) {
          const int k0 = t * 16 + gid, k1 = k0 + 8;
          if (k0 >= ntok || k0 < lead) u0 = 0u;
          if (k1 >= ntok || k1 < lead) u1 = 0u;
        }
        const float sA = h_lo(u0), sB = h_lo(u1);
        const float cA = fmaf(8.f, sA, h_hi(u0)), cB = fmaf(8.f, sB, h_hi(u1));   // min + 8 s
        uint32_t bh[NH][2], bl[NH][2];
#pragma unroll
        for (int nh = 0; nh < NH; ++nh) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float p0 = sc[t][nh][e], p1 = sc[t][nh][2 + e];
            cs[nh][e] = fmaf(p0, cA, fmaf(p1, cB, cs[nh][e]));
            sc[t][nh][e] = p0 * sA;
            sc[t][nh][2 + e] = p1 * sB;
          }
          // B fragments of P'^T (k = token, n = head): the S^T rows of tokens 0-7 / 8-15 of
          // the tile, packed per head pair and transposed
#pragma unroll
          for (int r = 0; r < 2; ++r) {
            const float x = sc[t][nh][2 * r], y = sc[t][nh][2 * r + 1];
            const uint32_t hi = pack_bf16(x, y);
            const uint32_t lo = pack_bf16(x - bf16_lo(hi), y - bf16_hi(hi));
            if (COMB) {
              const uint32_t lo_of_pair = __shfl_xor_sync(FULL_MASK, lo, 2);
              bh[nh][r] = movmatrix_t(tig < 2 ? hi : lo_of_pair);
            } else {
              bh[nh][r] = movmatrix_t(hi);
              bl[nh][r] = movmatrix_t(lo);
            }
          }
        }
        const int t0 = r0 + 2 * tig;                 // a0/a1: record rows t0, t0+1; a2/a3: +8
        const uint8_t* vc = st + T::VC + cv / 2;
#pragma unroll
        for (int w = 0; w < VW; ++w) {
          const uint32_t ra = *reinterpret_cast<const uint32_t*>(vc + (size_t)t0 * (D / 2) + 4 * w);
          const uint32_t rb = *reinterpret_cast<const uint32_t*>(vc + (size_t)(t0 + 1) * (D / 2) + 4 * w);
          const uint32_t rc = *reinterpret_cast<const uint32_t*>(vc + (size_t)(t0 + 8) * (D / 2) + 4 * w);
          const uint32_t rd = *reinterpret_cast<const uint32_t*>(vc + (size_t)(t0 + 9) * (D / 2) + 4 * w);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            // byte k of the two rows' words: [a_k, a_k, b_k, b_k]; the even nibble is fragment
            // row gid, the odd one row gid + 8
            const uint32_t sel = (uint32_t)k | ((uint32_t)k << 4) | ((uint32_t)(4 + k) << 8) | ((uint32_t)(4 + k) << 12);
            const uint32_t pab = prmt(ra, rb, sel), pcd = prmt(rc, rd, sel);
            uint32_t va[4];
            va[0] = v_codes8(pab);
            va[1] = v_codes8(pab >> 4);
            va[2] = v_codes8(pcd);
            va[3] = v_codes8(pcd >> 4);
#pragma unroll
            for (int nh = 0; nh < NH; ++nh) {
              mma_bf16(o[4 * w + k][nh], va, bh[nh][0], bh[nh][1]);
              if (!COMB) mma_bf16(o[4 * w + k][nh], va, bl[nh][0], bl[nh][1]);
            }
          }
        }
      }
    }

    if (flags & F_LAST) {
      float L[NH][2], C[NH][2];
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float x = l[nh][e], y = cs[nh][e];
#pragma unroll
          for (int msk = 4; msk < 32; msk <<= 1) {
            x += __shfl_xor_sync(FULL_MASK, x, msk);
            y += __shfl_xor_sync(FULL_MASK, y, msk);
          }
          L[nh][e] = x;
          C[nh][e] = y;
        }
      if (COMB) {                     // the high-part and low-part sums of O, added in both halves
#pragma unroll
        for (int md = 0; md < MD; ++md)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[md][0][i] += __shfl_xor_sync(FULL_MASK, o[md][0][i], 2);
      }
      const bool whole = flags & F_WHOLE;
      const long long part = (long long)s * a.n_kv + g + p;
#pragma unroll
      for (int nh = 0; nh < NH; ++nh)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int hl = hw0 + nh * 8 + 2 * tig + e;
          if (hl >= a.G) continue;
          const float inv = whole ? (L[nh][e] > 0.f ? 1.f / L[nh][e] : 0.f) : 1.f;
          const float c = C[nh][e];
          // m-tile md rows gid / gid+8 hold channel cv + 8*(md/4) + channel_of(2*(md%4) + 0 / 1)
          if (whole) {
            const size_t base = (qrow0 + hl) * D + cv;
#pragma unroll
            for (int md = 0; md < MD; ++md) {
              const int c0 = 8 * (md >> 2) + channel_of(2 * (md & 3)), c1 = 8 * (md >> 2) + channel_of(2 * (md & 3) + 1);
              if (a.out_f32) {
                float* out = reinterpret_cast<float*>(a.out) + base;
                out[c0] = (o[md][nh][e] + c) * inv;
                out[c1] = (o[md][nh][2 + e] + c) * inv;
              } else {
                __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(a.out) + base;
                out[c0] = __float2bfloat16_rn((o[md][nh][e] + c) * inv);
                out[c1] = __float2bfloat16_rn((o[md][nh][2 + e] + c) * inv);
              }
            }
          } else {
            float* wo = a.ws_o + ((size_t)part * a.G + hl) * D + cv;
#pragma unroll
            for (int md = 0; md < MD; ++md) {
              wo[8 * (md >> 2) + channel_of(2 * (md & 3))] = o[md][nh][e] + c;
              wo[8 * (md >> 2) + channel_of(2 * (md & 3) + 1)] = o[md][nh][2 + e] + c;
            }
            if (gid == 0)
              *reinterpret_cast<float2*>(a.ws_ml + ((size_t)part * a.G + hl) * 2) = make_float2(m[nh][e], L[nh][e]);
          }
        }
    }

    __syncwarp();
    if (MT > 1 && lane == 0) mbar_arrive(&empty[slot]);
    if (warp == 0 && pj < len) issue();
    if (++c_slot == S) {
      c_slot = 0;
      c_phase ^= 1u;
    }
    if (flags & F_END) break;
  }

  if (abort_flag && threadIdx.x == 0) {
    // let the copies of the stages issued but not consumed land before the CTA exits
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

template <int D, int BS, int NH, int MT, int TB, bool COMB>
static Int4Variant make_int4_variant() {
  Int4Variant v;
  v.fn = (const void*)decode_int4_kernel<D, BS, NH, MT, TB, COMB>;
  v.stages = ring_stages(TB * Int4Tile<D, BS>::STAGE, BS == 16 ? 11264 : 16384, "PKV_STAGES_INT4");
  v.smem = int4_smem_bytes<D, BS, TB>(v.stages);
  v.warps = MT;
  v.P = 0;
  return v;
}

// Kernel variant of a group of G heads: 0 = up to 4 heads (high and low parts in one n-tile),
// 1 = up to 8, 2 = up to 16, 3 = up to 32 (two warps), 4 = up to 64 (four warps).
static int int4_variant_index(int G) { return G <= 4 ? 0 : head_tiling(G) + 1; }

static Int4Variant* lookup_int4(int D, int BS, int vi) {
  static std::mutex mu;
  static Int4Variant table[2][3][5];
  static bool ready[2][3][5] = {};
  const int di = D == 128 ? 1 : 0, bi = BS == 16 ? 0 : (BS == 32 ? 1 : 2);
  std::lock_guard<std::mutex> lock(mu);
  Int4Variant& v = table[di][bi][vi];
  if (!ready[di][bi][vi]) {
#define PKV_V(d, b)                                                          \
  if (D == d && BS == b) {                                                   \
    if (vi == 0) v = make_int4_variant<d, b, 1, 1, b == 16 ? 2 : 1, true>(); \
    else if (vi == 1) v = make_int4_variant<d, b, 1, 1, b == 16 ? 2 : 1, false>(); \
    else if (vi == 2) v = make_int4_variant<d, b, 2, 1, 1, false>();        \
    else if (vi == 3) v = make_int4_variant<d, b, 2, 2, 1, false>();        \
    else v = make_int4_variant<d, b, 2, 4, 1, false>();                     \
  }
    PKV_V(64, 16) PKV_V(64, 32) PKV_V(64, 64) PKV_V(128, 16) PKV_V(128, 32) PKV_V(128, 64)
#undef PKV_V
    if (cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)v.smem) != cudaSuccess)
      return nullptr;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, v.fn, v.warps * 32, v.smem) != cudaSuccess || occ < 1)
      return nullptr;
    v.P = device_sm_count() * occ;
    ready[di][bi][vi] = true;
  }
  return &v;
}

int int4_pieces(int D, int BS, int G) {
  Int4Variant* v = lookup_int4(D, BS, int4_variant_index(G));
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

extern "C" size_t pkv_int4_record_bytes(int block_size, int head_dim) {
  if (head_dim != 64 && head_dim != 128) return 0;
  if (block_size != 16 && block_size != 32 && block_size != 64) return 0;
  return (size_t)block_size * head_dim + 4 * (size_t)head_dim + 4 * (size_t)block_size;
}

extern "C" pkv_status pkv_kv_quant_append_int4(const void* k, const void* v, const int64_t* slot_mapping,
                                               const int32_t* tail_seq, int n_tok, uint8_t* cache, void* k_tail,
                                               int tail_rows, int num_blocks, int block_size, int n_kv,
                                               int head_dim, int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_kv_quant_append_int4");
  if (n_tok < 0 || num_blocks < 0 || n_kv <= 0 || tail_rows < 0) return PKV_EINVAL;
  if (pkv_int4_record_bytes(block_size, head_dim) == 0) return PKV_EINVAL;
  if (n_tok == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !tail_seq || !cache || !k_tail) return PKV_EINVAL;
  if (!al16(k) || !al16(v) || !al16(cache) || !al16(k_tail)) return PKV_EINVAL;
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
  a.cache = cache;
  a.rec_bytes = pkv_int4_record_bytes(block_size, head_dim);
  a.k_tail = static_cast<__nv_bfloat16*>(k_tail);
  a.err = err_flag;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long warps = (long long)n_tok * n_kv;
  const long long qwarps = warps * (head_dim / 32);              // kKWarps per (token, kv head)
  const unsigned g1 = (unsigned)((qwarps * 32 + 255) / 256);
  const long long vecs = warps * (head_dim / 8);
  const unsigned g2 = (unsigned)((vecs + 255) / 256);
#define PKV_Q(d, b) \
  if (head_dim == d && block_size == b) quant_append_kernel<d, b><<<g1, 256, 0, st>>>(a);
  PKV_Q(128, 16) PKV_Q(128, 32) PKV_Q(128, 64) PKV_Q(64, 16) PKV_Q(64, 32) PKV_Q(64, 64)
#undef PKV_Q
  void* targs[] = {(void*)&a};
  cudaError_t e2 = launch_pdl(head_dim == 128 ? (const void*)tail_write_kernel<128> : (const void*)tail_write_kernel<64>,
                              dim3(g2), dim3(256), 0, st, targs);
  if (e2 != cudaSuccess) {
    record_cuda_error(e2);
    return PKV_ECUDA;
  }
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}

static pkv_status decode_int4(const void* q, const uint8_t* cache, const void* k_tail, const int32_t* block_tables,
                              int max_blocks,
                              const int32_t* context_lens, float scale, int window, int batch, int n_h, int n_kv,
                              int head_dim, int block_size, int num_blocks, void* out, int out_dtype, void* workspace,
                              size_t workspace_bytes, int32_t* err_flag, void* stream) {
  if (batch < 0 || !valid_shape(n_h, n_kv, head_dim, block_size) || max_blocks < 0 || num_blocks < 0 || window < 0)
    return PKV_EINVAL;
  if (out_dtype != PKV_OUT_BF16 && out_dtype != PKV_OUT_F32) return PKV_EINVAL;
  if (batch == 0) return PKV_OK;
  if (!q || !cache || !k_tail || !block_tables || !context_lens || !out || !workspace) return PKV_EINVAL;
  if (!al16(q) || !al16(cache) || !al16(k_tail) || !al16(out) || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PKV_EINVAL;
  if ((long long)max_blocks * block_size > 0x7fffffffLL) return PKV_ERANGE;
  const int G = n_h / n_kv;
  Int4Variant* vv = lookup_int4(head_dim, block_size, int4_variant_index(G));
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
  a.P_launch = vv->P;
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
  a.window = window;
  a.cache = cache;
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

extern "C" pkv_status pkv_paged_decode_attn_int4(const void* q, const uint8_t* cache, const void* k_tail,
                                                 const int32_t* block_tables, int max_blocks,
                                                 const int32_t* context_lens, float scale, int batch, int n_h,
                                                 int n_kv, int head_dim, int block_size, int num_blocks, void* out,
                                                 int out_dtype, void* workspace, size_t workspace_bytes,
                                                 int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_paged_decode_attn_int4");
  return decode_int4(q, cache, k_tail, block_tables, max_blocks, context_lens, scale, 0,
                     batch, n_h, n_kv, head_dim, block_size, num_blocks, out, out_dtype, workspace, workspace_bytes,
                     err_flag, stream);
}

extern "C" pkv_status pkv_paged_decode_attn_int4_window(const void* q, const uint8_t* cache, const void* k_tail,
                                                        const int32_t* block_tables,
                                                        int max_blocks, const int32_t* context_lens, float scale,
                                                        int window, int batch, int n_h, int n_kv, int head_dim,
                                                        int block_size, int num_blocks, void* out, int out_dtype,
                                                        void* workspace, size_t workspace_bytes, int32_t* err_flag,
                                                        void* stream) {
  PKV_NVTX("pkv_paged_decode_attn_int4_window");
  return decode_int4(q, cache, k_tail, block_tables, max_blocks, context_lens, scale, window, batch, n_h, n_kv, head_dim, block_size, num_blocks, out, out_dtype, workspace,
                     workspace_bytes, err_flag, stream);
}
