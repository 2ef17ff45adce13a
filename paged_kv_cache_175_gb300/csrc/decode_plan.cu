// Plan and split-reduce kernels of the paged decode attention, plus host utilities
// shared by every entry point (error bookkeeping, SM count, tensor-map encoding,
// programmatic-dependent launches).
#include <cudaTypedefs.h>

#include <atomic>
#include <cmath>
#include <cstdlib>
#include <mutex>

#include "decode_common.cuh"

namespace pkv {

static thread_local int g_last_cuda_error = 0;

void record_cuda_error(cudaError_t e) {
  if (e != cudaSuccess) g_last_cuda_error = (int)e;
}

int device_sm_count() {
  static std::atomic<int> cache[64];                          // zero-initialised (static storage)
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int n = cache[dev].load(std::memory_order_relaxed);
  if (!n) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

int encode_tensor_map_3d(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                         uint64_t stride1_bytes, uint64_t stride2_bytes, uint32_t box0, uint32_t box1) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!encode) return -1;
  const cuuint64_t dims[3] = {d0, d1, d2};
  const cuuint64_t strides[2] = {stride1_bytes, stride2_bytes};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t elem[3] = {1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
                      elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? 0 : (int)r;
}

int ring_stages(size_t stage_bytes, size_t ring_bytes, const char* env) {
  if (const char* e = getenv(env)) {
    const int v = atoi(e);
    if (v >= 2 && v <= 16) return v;
  }
  const int st = (int)(ring_bytes / stage_bytes);
  return st < 2 ? 2 : (st > 8 ? 8 : st);
}

cudaError_t launch_pdl(const void* func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       void** args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, func, args);
}

// ---- plan: range-check context lengths, scan blocks per sequence, start cursors ---------------
// One CTA.  The prefix sums also go to shared memory (up to kPlanSeqs sequences; beyond
// that the cursor search reads them back from global memory, which this CTA wrote), and
// every piece's start cursor is computed here so an attention CTA begins with one load.
constexpr int kPlanSeqs = 8192;

__global__ void __launch_bounds__(1024) plan_kernel(const int32_t* __restrict__ ctx, int batch, int max_ctx,
                                                    int block_size, int window, int n_kv, int P,
                                                    int32_t* __restrict__ cum,
                                                    int32_t* __restrict__ ctx_eff, int4* __restrict__ pieces,
                                                    int32_t* err) {
  __shared__ int warp_sums[32];
  __shared__ int carry;
  __shared__ int scum[kPlanSeqs + 1];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool in_smem = batch <= kPlanSeqs;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < batch; base += 1024) {
    const int s = base + threadIdx.x;
    int nb = 0;
    if (s < batch) {
      int c = ctx[s];
      if (c < 0 || c > max_ctx) {
        set_err(err, PKV_DEV_BAD_CTX);
        c = c < 0 ? 0 : max_ctx;
      }
      ctx_eff[s] = c;
      nb = span_blocks(c, window, block_size);
    }
    int x = nb;                                               // inclusive warp scan
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(FULL_MASK, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    const int excl = carry + (warp ? warp_sums[warp - 1] : 0) + x - nb;
    if (s < batch) {
      cum[s] = excl;
      if (in_smem) scum[s] = excl;
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry = excl + nb;
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    cum[batch] = carry;
    if (in_smem) scum[batch] = carry;
  }
  __syncthreads();
  const int* cu = in_smem ? scum : cum;
  const long long W = (long long)n_kv * carry;
  const int Pe = effective_pieces(W, P);
  for (int p = threadIdx.x; p < Pe; p += blockDim.x) {
    const long long pstart = W * p / Pe;
    if (pstart >= W) continue;                                // W == 0: nothing to start
    int lo = 0, hi = batch - 1;                               // largest s with n_kv * cum[s] <= pstart
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((long long)n_kv * cu[mid] <= pstart) lo = mid; else hi = mid - 1;
    }
    const int nb = cu[lo + 1] - cu[lo];
    const long long off = pstart - (long long)n_kv * cu[lo];
    pieces[2 * p] = make_int4(lo, (int)(off / nb), (int)(off % nb), nb);
    pieces[2 * p + 1] = make_int4(ctx_eff[lo], 0, 0, 0);
  }
}

cudaError_t launch_plan(const int32_t* context_lens, int batch, int max_ctx, int block_size,
                        const DecodeArgs& a, int P, cudaStream_t stream) {
  plan_kernel<<<1, 1024, 0, stream>>>(context_lens, batch, max_ctx, block_size, a.window, a.n_kv, P,
                                      const_cast<int32_t*>(a.cum), const_cast<int32_t*>(a.ctx_eff),
                                      const_cast<int4*>(a.pieces), a.err);
  return cudaGetLastError();
}

// ---- reduce: merge the partial softmax states of segments split across pieces ----------------
// The pieces a segment spans follow from the partition alone (the line of blocks and the
// attention grid's size), so every thread finds them before the grid-dependency wait, and
// the rows of segments that one piece holds (finished by the attention kernel itself) leave
// right after it.  Empty sequences get a zero row here.  Without a plan kernel the CTA first
// lays out the blocks of every sequence and their prefix sums in shared memory (one sequence
// per thread); the context lengths are inputs of the call, and the plan kernel's prefix sums
// finished before the attention kernel let this one launch.
//
// Two shapes.  Narrow, for batches whose segments span few pieces: LPR lanes per (sequence,
// q head) row -- a warp (8 rows per CTA), or half of one (16 rows per CTA, with half the loads
// per round) when a warp per row would take more CTAs than are resident at once.  Wide: one
// CTA per row whose eight warps take interleaved chunks of its pieces and combine their
// eight states through shared memory, for few long sequences, where a segment spans a large
// share of the grid's pieces and one warp would take one memory round trip per eight of them.

// Partial states a warp loads at a time in merge_pieces (LPR = 32 lanes per row: 8 per
// row; LPR = 16: 4 per row, two rows per warp).
constexpr int kMergeChunk = 8;

// Vector of V consecutive floats at src (V = 2, 4 or 8; 8-byte aligned, 16 for V >= 4).
template <int V>
__device__ __forceinline__ void load_vec(const float* src, float (&v)[V]) {
  if constexpr (V == 2) {
    const float2 x = *reinterpret_cast<const float2*>(src);
    v[0] = x.x; v[1] = x.y;
  } else {
#pragma unroll
    for (int j = 0; j < V / 4; ++j) {
      const float4 x = *reinterpret_cast<const float4*>(src + 4 * j);
      v[4 * j] = x.x; v[4 * j + 1] = x.y; v[4 * j + 2] = x.z; v[4 * j + 3] = x.w;
    }
  }
}

// Merges the states of pieces first, first+1, ... (chunks of CH taken every `step` pieces,
// none past p1) of one (segment, head) into the running (M, L, acc), base-2 exponents; the
// LPR lanes of the row hold V = D / LPR channels each (sub: the lane's place).  Every load of
// a chunk is issued before any is used, and chunks merge online.
template <int D, int LPR>
__device__ __forceinline__ void merge_pieces(const DecodeArgs& a, long long seg, int hl, int sub, int first,
                                             int p1, int step, float& M, float& L, float (&acc)[D / LPR]) {
  constexpr int V = D / LPR, CH = kMergeChunk * LPR / 32;
  for (int pc = first; pc <= p1; pc += step) {
    float mv[CH], lv[CH], ov[CH][V];
    bool use[CH];
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      const int p = pc + i;
      use[i] = p <= p1;
      mv[i] = -INFINITY;
      lv[i] = 0.f;
#pragma unroll
      for (int k = 0; k < V; ++k) ov[i][k] = 0.f;
      if (use[i]) {
        const long long part = (seg + p) * a.G + hl;
        const float2 ml = *reinterpret_cast<const float2*>(a.ws_ml + part * 2);
        mv[i] = ml.x;
        lv[i] = ml.y;
        load_vec<V>(a.ws_o + part * D + sub * V, ov[i]);
      }
    }
    float Mc = M;
#pragma unroll
    for (int i = 0; i < CH; ++i) Mc = fmaxf(Mc, mv[i]);
    const float r = ex2(M - Mc);                              // rescale what was merged so far
    L *= r;
#pragma unroll
    for (int k = 0; k < V; ++k) acc[k] *= r;
#pragma unroll
    for (int i = 0; i < CH; ++i) {
      if (!use[i]) continue;
      const float w = ex2(mv[i] - Mc);
      L += w * lv[i];
#pragma unroll
      for (int k = 0; k < V; ++k) acc[k] += w * ov[i][k];
    }
    M = Mc;
  }
}

// Wide reduce when the grid's pieces per segment reach this many (two chunks of the CTA).
constexpr int kWideReducePieces = 16;

template <int D, bool WIDE, int LPR>
__global__ void __launch_bounds__(256, LPR == 16 ? 4 : 0) reduce_kernel(const DecodeArgs a) {
  constexpr int V = D / LPR;                                  // channels per lane
  constexpr int RPC = 256 / LPR;                              // rows per CTA (narrow)
  static_assert(kInlinePlanSeqs == 8 * 32, "one sequence per thread of the CTA");
  static_assert(!WIDE || LPR == 32, "a wide CTA's warps each take the whole row");
  __shared__ int snb[kInlinePlanSeqs], spre[kInlinePlanSeqs], schunk[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = threadIdx.x % LPR;
  const int row = WIDE ? blockIdx.x : blockIdx.x * RPC + threadIdx.x / LPR;
  if (a.inline_plan) {
    // blocks of every sequence and their exclusive prefix: thread t takes sequence t
    const int sq = threadIdx.x;
    const int n = sq < a.batch ? span_blocks(clamp_ctx(a.ctx_raw[sq], a.max_ctx), a.window, a.block_size) : 0;
    int incl = n;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(FULL_MASK, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) schunk[warp] = incl;
    __syncthreads();
    int carry = 0;
    for (int c = 0; c < warp; ++c) carry += schunk[c];
    snb[sq] = n;
    spre[sq] = carry + incl - n;
    __syncthreads();
  }
  // Every thread passes the grid-dependency wait, also those with nothing to do: this grid
  // then completes only after the attention kernel, so no launch after it on the stream
  // can overlap that kernel.
  if (row >= a.batch * a.n_h) {
    grid_dep_wait();
    return;
  }
  const int s = row / a.n_h, hq = row % a.n_h, g = hq / a.G, hl = hq % a.G;
  const long long seg = (long long)s * a.n_kv + g;
  long long before, total;                                    // blocks of sequences < s, of all
  int nb;
  if (a.inline_plan) {
    before = spre[s];
    total = 0;
#pragma unroll
    for (int c = 0; c < 8; ++c) total += schunk[c];
    nb = snb[s];
  } else {
    before = a.cum[s];
    total = a.cum[a.batch];
    nb = a.cum[s + 1] - a.cum[s];
  }
  int p0 = 0, p1 = 0;
  if (nb > 0) {
    const long long W = (long long)a.n_kv * total;
    const int P = effective_pieces(W, a.P_launch);
    const long long start = (long long)a.n_kv * before + (long long)g * nb;
    p0 = piece_of(start, W, P);
    p1 = piece_of(start + nb - 1, W, P);
  }
  grid_dep_wait();
  if (nb > 0 && p0 == p1) return;                             // finished by the attention kernel
  // Every piece from p0 to p1 holds part of the segment (pieces hold at least 8 positions,
  // so none is empty) and wrote a state.
  float acc[V];
#pragma unroll
  for (int i = 0; i < V; ++i) acc[i] = 0.f;
  float M = -INFINITY, L = 0.f;
  if constexpr (WIDE) {
    __shared__ float sM[8], sL[8];
    __shared__ __align__(16) float sacc[8][D];
    if (nb > 0) merge_pieces<D, 32>(a, seg, hl, lane, p0 + warp * kMergeChunk, p1, 8 * kMergeChunk, M, L, acc);
    if constexpr (V == 4)
      *reinterpret_cast<float4*>(&sacc[warp][lane * V]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    else
      *reinterpret_cast<float2*>(&sacc[warp][lane * V]) = make_float2(acc[0], acc[1]);
    if (lane == 0) {
      sM[warp] = M;
      sL[warp] = L;
    }
    __syncthreads();
    // thread t < D/2 combines channels 2t, 2t+1 over the warps; warp 0 took p0, so the
    // largest exponent is finite and warps without pieces weigh zero
    const int t = threadIdx.x;
    if (t >= D / 2) return;
    float o0 = 0.f, o1 = 0.f;
    if (nb > 0) {
      float Mt = sM[0];
#pragma unroll
      for (int w = 1; w < 8; ++w) Mt = fmaxf(Mt, sM[w]);
      float Lt = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        const float f = ex2(sM[w] - Mt);
        Lt += f * sL[w];
        o0 += f * sacc[w][2 * t];
        o1 += f * sacc[w][2 * t + 1];
      }
      const float inv = Lt > 0.f ? 1.f / Lt : 0.f;
      o0 *= inv;
      o1 *= inv;
    }
    const size_t o = (size_t)row * D + 2 * t;
    if (a.out_f32) {
      *reinterpret_cast<float2*>(reinterpret_cast<float*>(a.out) + o) = make_float2(o0, o1);
    } else {
      *reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + o) = pack_bf16(o0, o1);
    }
  } else {
    if (nb > 0) {
      constexpr int CH = kMergeChunk * LPR / 32;
      merge_pieces<D, LPR>(a, seg, hl, sub, p0, p1, CH, M, L, acc);
      const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) acc[i] *= inv;
    }
    const size_t o = (size_t)row * D + sub * V;
    if (a.out_f32) {
      float* out = reinterpret_cast<float*>(a.out) + o;
#pragma unroll
      for (int i = 0; i < V; ++i) out[i] = acc[i];
    } else {
      uint32_t* out = reinterpret_cast<uint32_t*>(reinterpret_cast<__nv_bfloat16*>(a.out) + o);
#pragma unroll
      for (int i = 0; i < V / 2; ++i) out[i] = pack_bf16(acc[2 * i], acc[2 * i + 1]);
    }
  }
}

// CTAs of the warp-per-row reduce resident at once on the device (0 if the query failed).
static int reduce_wave() {
  int occ = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, reduce_kernel<128, false, 32>, 256, 0) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return occ * device_sm_count();
}

cudaError_t launch_reduce(int head_dim, const DecodeArgs& a, int P, cudaStream_t stream) {
  const int rows = a.batch * a.n_h;
  if (rows == 0) return cudaSuccess;
  // the grid's pieces over the segments: about the average a segment spans
  const bool wide = (long long)P >= (long long)kWideReducePieces * a.batch * a.n_kv;
  // Narrow: 16 lanes per row when a warp per row would take more CTAs than are resident at
  // once (the attention grid holds the SMs until it ends, so the CTAs past one wave would
  // start only after the first wave's merges).  Either shape gives the same result.
  static const int wave = reduce_wave();                      // one device per process
  const bool half = !wide && wave > 0 && (rows + 7) / 8 > wave;
  dim3 grid(wide ? rows : (half ? (rows + 15) / 16 : (rows + 7) / 8)), block(256);
  DecodeArgs args = a;
  void* kargs[] = {&args};
  const void* fn;
  if (head_dim == 128)
    fn = wide ? (const void*)reduce_kernel<128, true, 32>
              : (half ? (const void*)reduce_kernel<128, false, 16> : (const void*)reduce_kernel<128, false, 32>);
  else
    fn = wide ? (const void*)reduce_kernel<64, true, 32>
              : (half ? (const void*)reduce_kernel<64, false, 16> : (const void*)reduce_kernel<64, false, 32>);
  return launch_pdl(fn, grid, block, 0, stream, kargs);
}

// Self-test of the bounded wait every ring uses: one thread initialises an mbarrier for
// one arrival, arrives on it or not, and waits for the phase with a short limit.
__global__ void wait_selftest_kernel(int arrive, unsigned long long limit_ns, int32_t* err) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  if (arrive) mbar_arrive(&bar);
  if (!mbar_wait(&bar, 0, limit_ns)) set_err(err, PKV_DEV_TIMEOUT);
}

}  // namespace pkv

extern "C" const char* pkv_status_str(int status) {
  switch (status) {
    case PKV_OK: return "ok";
    case PKV_EINVAL: return "invalid argument";
    case PKV_ERANGE: return "size out of range";
    case PKV_ECUDA: return "CUDA error";
    case PKV_ENOSPC: return "workspace too small";
    default: return "unknown status";
  }
}

extern "C" int pkv_last_cuda_error(void) { return pkv::g_last_cuda_error; }

extern "C" pkv_status pkv_selftest_wait(int arrive, int limit_us, int32_t* err_flag, void* stream) {
  if (limit_us < 1 || limit_us > 2000000 || !err_flag) return PKV_EINVAL;
  pkv::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(arrive ? 1 : 0,
                                                                              1000ull * (unsigned long long)limit_us,
                                                                              err_flag);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    pkv::record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}

// Window of one layer from a per-layer list of attention windows that is repeated over the
// layers when it is shorter than the model.
extern "C" int pkv_layer_window(const int32_t* windows, int n, int layer) {
  if (!windows || n <= 0 || layer < 0) return -1;
  for (int i = 0; i < n; ++i)
    if (windows[i] <= 0) return -1;
  return windows[layer % n];
}
