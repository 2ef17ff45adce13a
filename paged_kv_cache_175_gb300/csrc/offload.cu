// Block copies between the GPU pools and host pools in page-locked memory: the data side
// of the block manager's offload and onload ("KV 캐시 시스템 (KV Cache System)", section
// "호스트 메모리로의 오프로딩").  The GPU reads and writes host memory directly (over
// NVLink-C2C on a GB300 node), 16-byte vectors, all loads of a thread in flight before its
// stores.  The host splits the recorded list into waves of independent copies.
#include <cstring>
#include <unordered_set>
#include <vector>

#include "../../include/pkv_bm.h"
#include "decode_common.cuh"   // record_cuda_error
#include "nvtx_range.h"

namespace pkv {

// Copies per launch, passed by value: (src, dst) with bit 31 of src set for an onload.
// 480 * 8 bytes keeps the parameter block under 4 KB.
constexpr int kCopiesPerLaunch = 480;
constexpr int kCopyThreads = 256;
constexpr int kVecPerThread = 4;                   // 16-byte vectors per thread per tensor
constexpr int kChunkBytes = kCopyThreads * kVecPerThread * 16;

struct CopyWave {
  int n;
  int2 op[kCopiesPerLaunch];
};

__global__ void __launch_bounds__(kCopyThreads)
    copy_blocks_kernel(const __grid_constant__ CopyWave w, uint4* __restrict__ k_pool, uint4* __restrict__ v_pool,
                       uint4* __restrict__ k_host, uint4* __restrict__ v_host, long long block_vecs) {
  const int i = blockIdx.y;
  if (i >= w.n) return;
  const int2 op = w.op[i];
  const bool onload = op.x < 0;
  const long long src = op.x & 0x7fffffff, dst = op.y;
  const uint4* ks = (onload ? k_host : k_pool) + src * block_vecs;
  const uint4* vs = (onload ? v_host : v_pool) + src * block_vecs;
  uint4* kd = (onload ? k_pool : k_host) + dst * block_vecs;
  uint4* vd = (onload ? v_pool : v_host) + dst * block_vecs;
  const long long base = (long long)blockIdx.x * (kCopyThreads * kVecPerThread) + threadIdx.x;
  uint4 a[kVecPerThread], b[kVecPerThread];
#pragma unroll
  for (int j = 0; j < kVecPerThread; ++j) {
    const long long e = base + (long long)j * kCopyThreads;
    if (e < block_vecs) {
      a[j] = ks[e];
      b[j] = vs[e];
    }
  }
#pragma unroll
  for (int j = 0; j < kVecPerThread; ++j) {
    const long long e = base + (long long)j * kCopyThreads;
    if (e < block_vecs) {
      kd[e] = a[j];
      vd[e] = b[j];
    }
  }
}

static bool gpu_addressable_host(const void* p) {
  cudaPointerAttributes at;
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost && at.devicePointer == p;
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_copy_blocks(const pkv_block_copy* copies, int n, void* k_pool, void* v_pool,
                                      int num_blocks, void* k_host, void* v_host, int host_blocks,
                                      size_t block_bytes, void* stream) {
  PKV_NVTX("pkv_copy_blocks");
  if (n < 0 || num_blocks < 0 || host_blocks < 0 || block_bytes == 0 || block_bytes % 16) return PKV_EINVAL;
  if (n == 0) return PKV_OK;
  if (!copies || !k_pool || !v_pool || !k_host || !v_host) return PKV_EINVAL;
  for (const void* p : {k_pool, v_pool, k_host, v_host})
    if (reinterpret_cast<uintptr_t>(p) & 15u) return PKV_EINVAL;
  for (int i = 0; i < n; ++i) {
    const pkv_block_copy& c = copies[i];
    if (c.kind == PKV_COPY_OFFLOAD) {
      if (c.src < 0 || c.src >= num_blocks || c.dst < 0 || c.dst >= host_blocks) return PKV_EINVAL;
    } else if (c.kind == PKV_COPY_ONLOAD) {
      if (c.src < 0 || c.src >= host_blocks || c.dst < 0 || c.dst >= num_blocks) return PKV_EINVAL;
    } else {
      return PKV_EINVAL;
    }
  }
  if (!gpu_addressable_host(k_host) || !gpu_addressable_host(v_host)) return PKV_EINVAL;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long long block_vecs = (long long)(block_bytes / 16);
  const unsigned chunks = (unsigned)((block_bytes + kChunkBytes - 1) / kChunkBytes);
  // waves: consecutive copies touching distinct GPU blocks and host slots
  std::unordered_set<int> gpu_used, host_used;
  CopyWave w;
  w.n = 0;
  auto flush = [&]() -> cudaError_t {
    if (w.n == 0) return cudaSuccess;
    copy_blocks_kernel<<<dim3(chunks, (unsigned)w.n), kCopyThreads, 0, st>>>(
        w, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), static_cast<uint4*>(k_host),
        static_cast<uint4*>(v_host), block_vecs);
    w.n = 0;
    return cudaGetLastError();
  };
  for (int i = 0; i < n; ++i) {
    const pkv_block_copy& c = copies[i];
    const int g = c.kind == PKV_COPY_OFFLOAD ? c.src : c.dst;
    const int h = c.kind == PKV_COPY_OFFLOAD ? c.dst : c.src;
    cudaError_t e = cudaSuccess;
    if (gpu_used.count(g) || host_used.count(h)) {     // depends on an earlier copy: new wave
      e = flush();
      gpu_used.clear();
      host_used.clear();
    } else if (w.n == kCopiesPerLaunch) {
      e = flush();                                     // same wave, next launch
    }
    if (e != cudaSuccess) {
      record_cuda_error(e);
      return PKV_ECUDA;
    }
    gpu_used.insert(g);
    host_used.insert(h);
    w.op[w.n++] = make_int2(c.kind == PKV_COPY_ONLOAD ? (int)(0x80000000u | (unsigned)c.src) : c.src, c.dst);
  }
  const cudaError_t e = flush();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}
