// CacheBlend's model-free steps on the paged cache ("Research Paper Review : CACHE BLEND
// ...", sections "Methods" and "System Design"): the KV deviation of each candidate token
// between its reused (precomputed) K/V in the pool and its recomputed K/V, the selection
// of the tokens with the largest deviation, and the fuse that writes the recomputed rows
// of the selected tokens into the cache.
#include <cmath>

#include "../../include/pkv.h"
#include "decode_common.cuh"
#include "nvtx_range.h"

namespace pkv {

// ---- deviation: a group of lanes per token, 16-byte vectors, every load of a pass in flight --
// A token's K and V rows (n_kv * head_dim / 8 vectors each) go to `lpt` lanes, the
// smallest power of two covering them, at most 32; a warp takes 32 / lpt tokens at once.
constexpr int kDevThreads = 256;

__host__ __device__ inline int dev_lanes_per_token(int vec_per_tok) {
  int l = 4;
  while (l < 32 && l < vec_per_tok) l <<= 1;
  return l;
}

// Rows of at most `lpt` vectors (one vector per lane and tensor: n_kv * head_dim <= 256,
// the MQA shapes): each lane group takes kDevTok tokens per pass, with every slot load, then
// every data load of the pass issued before any is used -- four times the bytes in flight
// of one token per pass, which a short row leaves too few of to cover the memory latency.
constexpr int kDevTok = 4;

__global__ void __launch_bounds__(kDevThreads)
    kv_deviation_short_kernel(const uint4* __restrict__ k_pool, const uint4* __restrict__ v_pool,
                              const int64_t* __restrict__ slots, const uint4* __restrict__ k_new,
                              const uint4* __restrict__ v_new, long long n, int n_kv, int block_size,
                              int vec_per_row, long long n_slots, int bs_shift, int vpr_shift, float* __restrict__ dev,
                              int32_t* err) {
  grid_dep_launch();                       // a following selection may launch; it waits for this grid
  const int lane = threadIdx.x & 31;
  const int vec_per_tok = n_kv * vec_per_row;
  const int lpt = dev_lanes_per_token(vec_per_tok), tpw = 32 / lpt;
  const int sub = lane / lpt, sl = lane % lpt;
  const long long groups = (long long)gridDim.x * (kDevThreads / 32) * tpw;
  const long long gq = (blockIdx.x * (long long)(kDevThreads / 32) + (threadIdx.x >> 5)) * tpw + sub;
  const bool has_vec = sl < vec_per_tok;
  int g = 0, w = sl;
  if (has_vec) {
    g = vpr_shift >= 0 ? sl >> vpr_shift : sl / vec_per_row;
    w = sl - g * vec_per_row;
  }
  for (long long base = 0; base < n; base += kDevTok * groups) {   // the same passes in every lane
    long long slot[kDevTok];
    bool live[kDevTok], bad[kDevTok];
    uint4 a[kDevTok], b[kDevTok], c[kDevTok], d[kDevTok];
#pragma unroll
    for (int u = 0; u < kDevTok; ++u) {                 // slots and recomputed rows (independent)
      const long long t = base + u * groups + gq;
      slot[u] = t < n ? slots[t] : 0;
      if (t < n && has_vec) {
        c[u] = __ldg(k_new + t * vec_per_tok + sl);
        d[u] = __ldg(v_new + t * vec_per_tok + sl);
      }
    }
#pragma unroll
    for (int u = 0; u < kDevTok; ++u) {                 // then the cached rows the slots point at
      const long long t = base + u * groups + gq;
      bad[u] = t < n && (slot[u] < 0 || slot[u] >= n_slots);
      live[u] = t < n && !bad[u];
      if (live[u] && has_vec) {
        const long long blk = bs_shift >= 0 ? slot[u] >> bs_shift : slot[u] / block_size;
        const long long row = slot[u] - blk * block_size;
        const size_t src = (((size_t)blk * n_kv + g) * block_size + row) * vec_per_row + w;
        a[u] = __ldg(k_pool + src);
        b[u] = __ldg(v_pool + src);
      }
    }
#pragma unroll
    for (int u = 0; u < kDevTok; ++u) {
      float acc = 0.f;
      if (live[u] && has_vec) {
        const uint32_t* pa = reinterpret_cast<const uint32_t*>(&a[u]);
        const uint32_t* pb = reinterpret_cast<const uint32_t*>(&b[u]);
        const uint32_t* pc = reinterpret_cast<const uint32_t*>(&c[u]);
        const uint32_t* pd = reinterpret_cast<const uint32_t*>(&d[u]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float k0 = bf16_lo(pa[j]) - bf16_lo(pc[j]), k1 = bf16_hi(pa[j]) - bf16_hi(pc[j]);
          const float v0 = bf16_lo(pb[j]) - bf16_lo(pd[j]), v1 = bf16_hi(pb[j]) - bf16_hi(pd[j]);
          acc = fmaf(k0, k0, acc);
          acc = fmaf(k1, k1, acc);
          acc = fmaf(v0, v0, acc);
          acc = fmaf(v1, v1, acc);
        }
      }
      for (int o = lpt / 2; o; o >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, o);   // within the group
      const long long t = base + u * groups + gq;
      if (sl == 0 && t < n) {
        if (bad[u]) set_err(err, PKV_DEV_BAD_SLOT);
        dev[t] = bad[u] ? 0.f : sqrtf(acc);
      }
    }
  }
}

__global__ void __launch_bounds__(kDevThreads)
    kv_deviation_kernel(const uint4* __restrict__ k_pool, const uint4* __restrict__ v_pool,
                        const int64_t* __restrict__ slots, const uint4* __restrict__ k_new,
                        const uint4* __restrict__ v_new, long long n, int n_kv, int block_size, int vec_per_row,
                        long long n_slots, int bs_shift, int vpr_shift, float* __restrict__ dev, int32_t* err) {
  // bs_shift / vpr_shift: log2 of block_size / vec_per_row when they are powers of two
  // (every shape the attention kernels take), else -1 and the index math divides
  grid_dep_launch();                       // a following selection may launch; it waits for this grid
  const int lane = threadIdx.x & 31;
  const int vec_per_tok = n_kv * vec_per_row;
  const int lpt = dev_lanes_per_token(vec_per_tok), tpw = 32 / lpt;
  const int sub = lane / lpt, sl = lane % lpt;
  const long long step = (long long)gridDim.x * (kDevThreads / 32) * tpw;
  for (long long t0 = (blockIdx.x * (long long)(kDevThreads / 32) + (threadIdx.x >> 5)) * tpw; t0 < n;
       t0 += step) {
    const long long t = t0 + sub;
    const long long slot = t < n ? slots[t] : 0;
    const bool bad = t < n && (slot < 0 || slot >= n_slots);
    const bool live = t < n && !bad;
    long long blk = 0, row = 0;
    if (live) {
      blk = bs_shift >= 0 ? slot >> bs_shift : slot / block_size;
      row = slot - blk * block_size;
    }
    const uint4* kn = k_new + (live ? t : 0) * vec_per_tok;
    const uint4* vn = v_new + (live ? t : 0) * vec_per_tok;
    float acc = 0.f;
    for (int base = 0; base < vec_per_tok; base += 2 * lpt) {
      uint4 a[2], b[2], c[2], d[2];
      bool ok[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int i = base + u * lpt + sl;
        ok[u] = live && i < vec_per_tok;
        if (ok[u]) {
          const int g = vpr_shift >= 0 ? i >> vpr_shift : i / vec_per_row, w = i - g * vec_per_row;
          const size_t src = (((size_t)blk * n_kv + g) * block_size + row) * vec_per_row + w;
          a[u] = __ldg(k_pool + src);
          b[u] = __ldg(v_pool + src);
          c[u] = __ldg(kn + i);
          d[u] = __ldg(vn + i);
        }
      }
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        if (!ok[u]) continue;
        const uint32_t* pa = reinterpret_cast<const uint32_t*>(&a[u]);
        const uint32_t* pb = reinterpret_cast<const uint32_t*>(&b[u]);
        const uint32_t* pc = reinterpret_cast<const uint32_t*>(&c[u]);
        const uint32_t* pd = reinterpret_cast<const uint32_t*>(&d[u]);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float k0 = bf16_lo(pa[j]) - bf16_lo(pc[j]), k1 = bf16_hi(pa[j]) - bf16_hi(pc[j]);
          const float v0 = bf16_lo(pb[j]) - bf16_lo(pd[j]), v1 = bf16_hi(pb[j]) - bf16_hi(pd[j]);
          acc = fmaf(k0, k0, acc);
          acc = fmaf(k1, k1, acc);
          acc = fmaf(v0, v0, acc);
          acc = fmaf(v1, v1, acc);
        }
      }
    }
    for (int o = lpt / 2; o; o >>= 1) acc += __shfl_xor_sync(FULL_MASK, acc, o);   // within the group
    if (sl == 0 && t < n) {
      if (bad) set_err(err, PKV_DEV_BAD_SLOT);
      dev[t] = bad ? 0.f : sqrtf(acc);
    }
  }
}

// ---- selection: one CTA per segment, radix select of the k-th largest key ------------------
// Key of element i of a segment: the order-preserving 32-bit image of its float value in
// the high half, the complement of i in the low half, so keys are distinct and a larger
// key means a larger value or, for equal values, a smaller index.
constexpr int kSelThreads = 1024;

__device__ __forceinline__ uint32_t float_order(float x) {
  const uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ unsigned long long sel_key(const float* dev, int i) {
  return ((unsigned long long)float_order(dev[i]) << 32) | (uint32_t)~(uint32_t)i;
}

// Exclusive scan of one int per thread over the CTA; returns this thread's prefix and
// writes the total to *total (kSelThreads threads).
__device__ __forceinline__ int cta_exclusive_scan(int x, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(FULL_MASK, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) warp_tot[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = warp_tot[lane];
    int wi = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, wi, o);
      if (lane >= o) wi += y;
    }
    warp_tot[lane] = wi - w;                                   // exclusive warp offsets
    if (lane == 31) *total = wi;
  }
  __syncthreads();
  const int r = warp_tot[warp] + incl - x;
  __syncthreads();
  return r;
}

__global__ void __launch_bounds__(kSelThreads)
    select_top_kernel(const float* __restrict__ dev, const int32_t* __restrict__ seg_offsets,
                      const int32_t* __restrict__ counts, int n_seg, int32_t* __restrict__ out) {
  __shared__ int hist[256];
  __shared__ int warp_tot[32];
  __shared__ int total;
  __shared__ unsigned long long prefix_sh;
  __shared__ int remain_sh, done_sh;
  grid_dep_wait();                         // the deviations come from the kernel before this one
  grid_dep_launch();
  const int s = blockIdx.x;
  const int lo = seg_offsets[s], hi = seg_offsets[s + 1];
  const int n = hi > lo ? hi - lo : 0;
  int k = counts[s];
  k = k < 0 ? 0 : (k > n ? n : k);
  // output base: the counts of the segments before this one (each clamped the same way)
  int base = 0;
  for (int j = threadIdx.x; j < s; j += kSelThreads) {
    const int nj = seg_offsets[j + 1] - seg_offsets[j];
    const int kj = counts[j];
    base += kj < 0 ? 0 : (kj > (nj > 0 ? nj : 0) ? (nj > 0 ? nj : 0) : kj);
  }
  base = cta_exclusive_scan(base, warp_tot, &total);
  base = total;
  if (k == 0) return;
  const float* d = dev + lo;
  // a segment of at most one key per thread keeps its keys in registers for every pass
  const bool held = n <= kSelThreads;
  const unsigned long long mine = held && (int)threadIdx.x < n ? sel_key(d, threadIdx.x) : 0ull;
  unsigned long long thresh = 0;                               // keys >= thresh are selected
  if (k < n) {
    // most significant byte first: find the byte of the k-th largest key, pass by pass;
    // stop early once the bin holding it is taken whole (then every key at or above the
    // prefix is selected)
    unsigned long long prefix = 0;
    int remain = k;
    for (int pass = 0; pass < 8; ++pass) {
      const int shift = 56 - 8 * pass;
      const unsigned long long hmask = pass == 0 ? 0ull : (~0ull << (shift + 8));
      for (int j = threadIdx.x; j < 256; j += kSelThreads) hist[j] = 0;
      __syncthreads();
      for (int i = threadIdx.x; i < n; i += kSelThreads) {
        const unsigned long long key = held ? mine : sel_key(d, i);
        if ((key & hmask) == prefix) atomicAdd(&hist[(key >> shift) & 255], 1);
      }
      __syncthreads();
      if (threadIdx.x < 32) {
        // lane l holds bins 255-8l down to 248-8l; counts from the top bin downwards
        const int lane = threadIdx.x;
        int c[8], tot = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          c[u] = hist[255 - 8 * lane - u];
          tot += c[u];
        }
        int incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(FULL_MASK, incl, o);
          if (lane >= o) incl += y;
        }
        int above = incl - tot;                             // keys in higher bins
        // the lane whose bins take the cumulative count to `remain` holds the k-th key
        // (bin 0 of lane 31 catches whatever is left)
        if (above < remain && (incl >= remain || lane == 31)) {
          int b = 255 - 8 * lane;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (above + c[u] >= remain || (lane == 31 && u == 7)) {
              b = 255 - 8 * lane - u;
              remain_sh = remain - above;
              done_sh = (c[u] == remain - above) ? 1 : 0;
              prefix_sh = prefix | ((unsigned long long)b << shift);
              break;
            }
            above += c[u];
          }
        }
      }
      __syncthreads();
      prefix = prefix_sh;
      remain = remain_sh;
      const int done = done_sh;
      __syncthreads();
      if (done) break;
    }
    thresh = prefix;                       // the k-th largest key, or the prefix of its whole bin
  }
  // compaction in index order
  int written = 0;
  for (int c0 = 0; c0 < n; c0 += kSelThreads) {
    const int i = c0 + threadIdx.x;
    const int f = (i < n && (k == n || (held ? mine : sel_key(d, i)) >= thresh)) ? 1 : 0;
    const int pos = cta_exclusive_scan(f, warp_tot, &total);
    if (f) out[base + written + pos] = lo + i;
    written += total;
    __syncthreads();
  }
}

// ---- fuse: recomputed rows of the selected tokens into the pools ----------------------------
__global__ void __launch_bounds__(256) kv_fuse_kernel(const uint4* __restrict__ k_new, const uint4* __restrict__ v_new,
                                                      const int64_t* __restrict__ row_slots,
                                                      const int32_t* __restrict__ rows, long long total,
                                                      int vec_per_row, int n_kv, int block_size, long long n_slots,
                                                      long long n_rows, uint4* __restrict__ k_pool,
                                                      uint4* __restrict__ v_pool, int32_t* err) {
  grid_dep_wait();                         // the selected rows come from the kernel before this one
  const int vec_per_tok = vec_per_row * n_kv;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long j = idx / vec_per_tok;
    const int e = (int)(idx - j * vec_per_tok);
    const int g = e / vec_per_row, vec = e - g * vec_per_row;
    const long long r = rows[j];
    const long long slot = (r >= 0 && r < n_rows) ? row_slots[r] : -1;
    if (slot < 0 || slot >= n_slots) {
      if (e == 0) set_err(err, PKV_DEV_BAD_SLOT);
      continue;
    }
    const long long blk = slot / block_size, off = slot - blk * block_size;
    const size_t dst = (((size_t)blk * n_kv + g) * block_size + off) * vec_per_row + vec;
    k_pool[dst] = k_new[r * vec_per_tok + e];
    v_pool[dst] = v_new[r * vec_per_tok + e];
  }
}

}  // namespace pkv

using namespace pkv;

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static int log2_if_pow2(int x) {
  if (x <= 0 || (x & (x - 1))) return -1;
  int k = 0;
  while ((1 << k) < x) ++k;
  return k;
}

extern "C" pkv_status pkv_kv_deviation(const void* k_pool, const void* v_pool, const int64_t* slots,
                                       const void* k_new, const void* v_new, int n, int num_blocks, int block_size,
                                       int n_kv, int head_dim, float* dev, int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_kv_deviation");
  if (n < 0 || num_blocks < 0 || block_size < 1 || n_kv < 1 || head_dim < 8 || head_dim % 8) return PKV_EINVAL;
  if (n == 0) return PKV_OK;
  if (!k_pool || !v_pool || !slots || !k_new || !v_new || !dev) return PKV_EINVAL;
  if (!al16(k_pool) || !al16(v_pool) || !al16(k_new) || !al16(v_new)) return PKV_EINVAL;
  const int vpr = head_dim / 8;
  const int tokens_per_cta = kDevThreads / 32 * (32 / dev_lanes_per_token(n_kv * vpr));
  if (n_kv * vpr <= dev_lanes_per_token(n_kv * vpr)) {
    // one vector per lane and tensor: kDevTok tokens per lane group and pass
    // a persistent grid of the CTAs that fit at once (two per SM at this kernel's registers);
    // the lanes loop over passes
    const long long want = ((long long)n + tokens_per_cta * kDevTok - 1) / (tokens_per_cta * kDevTok);
    const int grid = (int)(want < 2LL * device_sm_count() ? want : 2LL * device_sm_count());
    kv_deviation_short_kernel<<<grid, kDevThreads, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint4*>(k_pool), static_cast<const uint4*>(v_pool), slots,
        static_cast<const uint4*>(k_new), static_cast<const uint4*>(v_new), n, n_kv, block_size, vpr,
        (long long)num_blocks * block_size, log2_if_pow2(block_size), log2_if_pow2(vpr), dev, err_flag);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return PKV_ECUDA;
    }
    return PKV_OK;
  }
  const long long want = ((long long)n + tokens_per_cta - 1) / tokens_per_cta;
  const int grid = (int)(want < 16LL * device_sm_count() ? want : 16LL * device_sm_count());
  kv_deviation_kernel<<<grid, kDevThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k_pool), static_cast<const uint4*>(v_pool), slots, static_cast<const uint4*>(k_new),
      static_cast<const uint4*>(v_new), n, n_kv, block_size, vpr, (long long)num_blocks * block_size,
      log2_if_pow2(block_size), log2_if_pow2(vpr), dev, err_flag);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}

extern "C" pkv_status pkv_select_top(const float* dev, const int32_t* seg_offsets, const int32_t* counts, int n_seg,
                                     int32_t* out, void* stream) {
  PKV_NVTX("pkv_select_top");
  if (n_seg < 0) return PKV_EINVAL;
  if (n_seg == 0) return PKV_OK;
  if (!dev || !seg_offsets || !counts || !out) return PKV_EINVAL;
  void* args[] = {(void*)&dev, (void*)&seg_offsets, (void*)&counts, (void*)&n_seg, (void*)&out};
  const cudaError_t e = launch_pdl((const void*)select_top_kernel, dim3(n_seg), dim3(kSelThreads), 0,
                                   static_cast<cudaStream_t>(stream), args);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}

extern "C" pkv_status pkv_kv_fuse(const void* k_new, const void* v_new, const int64_t* row_slots, int n_rows,
                                  const int32_t* rows, int n_sel, void* k_pool, void* v_pool, int num_blocks,
                                  int block_size, int n_kv, int head_dim, int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_kv_fuse");
  if (n_sel < 0 || n_rows < 0 || num_blocks < 0 || block_size < 1 || n_kv < 1 || head_dim < 8 || head_dim % 8)
    return PKV_EINVAL;
  if (n_sel == 0) return PKV_OK;
  if (!k_new || !v_new || !rows || !row_slots || !k_pool || !v_pool) return PKV_EINVAL;
  if (!al16(k_new) || !al16(v_new) || !al16(k_pool) || !al16(v_pool)) return PKV_EINVAL;
  const int vpr = head_dim / 8;
  const long long total = (long long)n_sel * n_kv * vpr;
  const long long want = (total + 255) / 256;
  const int grid = (int)(want < 32LL * device_sm_count() ? want : 32LL * device_sm_count());
  const uint4* kn = static_cast<const uint4*>(k_new);
  const uint4* vn = static_cast<const uint4*>(v_new);
  uint4* kp = static_cast<uint4*>(k_pool);
  uint4* vp = static_cast<uint4*>(v_pool);
  long long n_slots = (long long)num_blocks * block_size, rows_ll = n_rows;
  void* args[] = {(void*)&kn, (void*)&vn, (void*)&row_slots, (void*)&rows, (void*)&total, (void*)&vpr,
                  (void*)&n_kv, (void*)&block_size, (void*)&n_slots, (void*)&rows_ll, (void*)&kp, (void*)&vp,
                  (void*)&err_flag};
  const cudaError_t e = launch_pdl((const void*)kv_fuse_kernel, dim3(grid), dim3(256), 0,
                                   static_cast<cudaStream_t>(stream), args);
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}

extern "C" double pkv_recompute_ratio(double load_time, double full_recompute_time) {
  double r = full_recompute_time > 0.0 ? load_time / full_recompute_time : 1.0;
  if (!(r >= 0.15)) r = 0.15;                                  // also catches NaN
  return r > 1.0 ? 1.0 : r;
}

extern "C" int pkv_select_count(double ratio, int n) {
  if (n <= 0 || !(ratio > 0.0)) return 0;
  const double x = ratio * (double)n - 1e-12;
  const int k = (int)std::ceil(x);
  return k < 0 ? 0 : (k > n ? n : k);
}
