// KV append (bf16 scatter by slot) and RoPE re-rotation of reused key blocks.
#include <cmath>

#include "decode_common.cuh"
#include "nvtx_range.h"

namespace pkv {

// One thread per 16-byte vector of one (token, kv head) row: loads and stores are
// coalesced along head_dim, and each (token, head) row lands as one contiguous run.
__global__ void __launch_bounds__(256) kv_append_kernel(const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                        const int64_t* __restrict__ slots, long long total,
                                                        int vec_per_row, int n_kv, int block_size,
                                                        long long n_slots, uint4* __restrict__ k_pool,
                                                        uint4* __restrict__ v_pool, int32_t* err) {
  grid_dep_launch();                       // the attention's setup may overlap this kernel
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const long long row = idx / vec_per_row;                  // (token, head)
    const int vec = (int)(idx - row * vec_per_row);
    const long long tok = row / n_kv;
    const int g = (int)(row - tok * n_kv);
    const long long slot = slots[tok];
    if (slot < 0) continue;
    if (slot >= n_slots) {
      if (g == 0 && vec == 0) set_err(err, PKV_DEV_BAD_SLOT);
      continue;
    }
    const long long blk = slot / block_size, off = slot - blk * block_size;
    const size_t dst = (((size_t)blk * n_kv + g) * block_size + off) * vec_per_row + vec;
    k_pool[dst] = k[idx];
    v_pool[dst] = v[idx];
  }
}

// One CTA per listed block.  Angles delta * inv_freq[j] are formed in fp64, reduced
// to [-pi, pi] in fp64 (k = rint(angle / 2pi)), and only the reduced angle goes to
// the fp32 sincos, so large position deltas keep full fp32 accuracy.  The rotation
// itself runs in fp32 on bf16 pairs and stores with round-to-nearest-even.
struct RopeFreq {
  double inv_freq[64];
};

template <int D>
__global__ void __launch_bounds__(256) rope_shift_kernel(__nv_bfloat16* __restrict__ k_pool,
                                                         const int32_t* __restrict__ block_ids,
                                                         const int32_t* __restrict__ deltas, int num_blocks,
                                                         int n_kv, int block_size, const RopeFreq f, int32_t* err) {
  constexpr int H = D / 2;
  __shared__ float cs[H], sn[H];
  const int phys = block_ids[blockIdx.x];
  const int delta = deltas[blockIdx.x];
  if ((unsigned)phys >= (unsigned)num_blocks) {
    if (threadIdx.x == 0) set_err(err, PKV_DEV_BAD_BLOCK);
    return;
  }
  if (delta == 0) return;                                     // rotation by 0 is the identity
  const double two_pi = 6.283185307179586476925286766559;
  for (int j = threadIdx.x; j < H; j += blockDim.x) {
    const double ang = (double)delta * f.inv_freq[j];
    const double r = ang - rint(ang / two_pi) * two_pi;
    float sv, cv;
    sincosf((float)r, &sv, &cv);
    cs[j] = cv;
    sn[j] = sv;
  }
  __syncthreads();
  const int rows = n_kv * block_size;
  // one 16-byte vector of each half of a row per item: channels j0..j0+7 and their partners
  constexpr int V = H / 8;                                    // vectors per half row
  uint4* base = reinterpret_cast<uint4*>(k_pool + (size_t)phys * rows * D);
  for (int idx = threadIdx.x; idx < rows * V; idx += blockDim.x) {
    const int r = idx / V, v = idx - r * V;
    uint4* row = base + (size_t)r * (D / 8);
    uint4 a = row[v], b = row[v + V];
    const int j0 = 8 * v;
    auto rot = [&](uint32_t& wa, uint32_t& wb, int j) {     // channels j, j + 1 and j + H, j + H + 1
      const float x1a = bf16_lo(wa), x1b = bf16_hi(wa), x2a = bf16_lo(wb), x2b = bf16_hi(wb);
      const float y1a = x1a * cs[j] - x2a * sn[j], y1b = x1b * cs[j + 1] - x2b * sn[j + 1];
      const float y2a = x1a * sn[j] + x2a * cs[j], y2b = x1b * sn[j + 1] + x2b * cs[j + 1];
      wa = pack_bf16(y1a, y1b);
      wb = pack_bf16(y2a, y2b);
    };
    rot(a.x, b.x, j0);
    rot(a.y, b.y, j0 + 2);
    rot(a.z, b.z, j0 + 4);
    rot(a.w, b.w, j0 + 6);
    row[v] = a;
    row[v + V] = b;
  }
}

}  // namespace pkv

using namespace pkv;

static bool al16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

extern "C" pkv_status pkv_kv_append(const void* k, const void* v, const int64_t* slot_mapping, int n_tok,
                                    void* k_pool, void* v_pool, int num_blocks, int block_size, int n_kv,
                                    int head_dim, int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_kv_append");
  if (n_tok < 0 || num_blocks < 0 || block_size <= 0 || n_kv <= 0) return PKV_EINVAL;
  if (head_dim != 64 && head_dim != 128) return PKV_EINVAL;
  if (block_size != 16 && block_size != 32 && block_size != 64) return PKV_EINVAL;
  if (n_tok == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_pool || !v_pool) return PKV_EINVAL;
  if (!al16(k) || !al16(v) || !al16(k_pool) || !al16(v_pool)) return PKV_EINVAL;
  const int vec = head_dim / 8;
  const long long total = (long long)n_tok * n_kv * vec;
  const int threads = 256;
  long long blocks = (total + threads - 1) / threads;
  const int cap = device_sm_count() > 0 ? device_sm_count() * 16 : 2048;
  if (blocks > cap) blocks = cap;
  kv_append_kernel<<<(unsigned)blocks, threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(k), static_cast<const uint4*>(v), slot_mapping, total, vec, n_kv, block_size,
      (long long)num_blocks * block_size, static_cast<uint4*>(k_pool), static_cast<uint4*>(v_pool), err_flag);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}

extern "C" pkv_status pkv_rope_shift_k(void* k_pool, const int32_t* block_ids, const int32_t* deltas, int n_blocks,
                                       int num_blocks, int n_kv, int block_size, int head_dim, double rope_base,
                                       int32_t* err_flag, void* stream) {
  PKV_NVTX("pkv_rope_shift_k");
  if (n_blocks < 0 || num_blocks < 0 || n_kv <= 0) return PKV_EINVAL;
  if (head_dim != 64 && head_dim != 128) return PKV_EINVAL;
  if (block_size != 16 && block_size != 32 && block_size != 64) return PKV_EINVAL;
  if (!(rope_base > 0.0) || !std::isfinite(rope_base)) return PKV_EINVAL;
  if (n_blocks == 0) return PKV_OK;
  if (!k_pool || !block_ids || !deltas || !al16(k_pool)) return PKV_EINVAL;
  RopeFreq f = {};
  for (int j = 0; j < head_dim / 2; ++j) f.inv_freq[j] = std::pow(rope_base, -2.0 * j / head_dim);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // one thread per 16-byte vector pair of a block, at most 256 (they loop), at least 64
  const long long items = (long long)n_kv * block_size * (head_dim / 16);
  const int threads = items >= 256 ? 256 : (items <= 64 ? 64 : (int)((items + 31) / 32 * 32));
  if (head_dim == 128)
    rope_shift_kernel<128><<<n_blocks, threads, 0, st>>>(static_cast<__nv_bfloat16*>(k_pool), block_ids, deltas,
                                                         num_blocks, n_kv, block_size, f, err_flag);
  else
    rope_shift_kernel<64><<<n_blocks, threads, 0, st>>>(static_cast<__nv_bfloat16*>(k_pool), block_ids, deltas,
                                                        num_blocks, n_kv, block_size, f, err_flag);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}
