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

// The listed blocks' rows are cut into equal ranges of ipc items (an item: one 16-byte
// vector of each half of a row, 32 bytes), about 32 KB per CTA: several consecutive listed
// blocks when blocks are small, part of one (or of two) when they are large.  Every thread
// issues all of its loads (NI items) before the angle tables are built, so the loads and
// the fp64 / sincos work overlap and a CTA needs one memory round trip.  Angles
// delta * inv_freq[j] are formed in fp64 and reduced to [-pi, pi] in fp64
// (k = rint(angle / 2pi), taken as a product with 1 / 2pi), and only the reduced angle goes
// to the fp32 sincos, so large position deltas keep full fp32 accuracy.  A block whose
// delta equals its predecessor's in the CTA reuses its table (the blocks of a reused chunk
// share one delta).  The rotation runs in fp32 on bf16 pairs and stores with
// round-to-nearest-even.
struct RopeFreq {
  double inv_freq[64];
};
constexpr int kRopeMaxBPC = 8;      // blocks a CTA's range may touch
constexpr int kRopeNI = 4;          // items per thread and round (64 registers: 4 CTAs per SM)

template <int D>
__global__ void __launch_bounds__(256, 4) rope_shift_kernel(__nv_bfloat16* __restrict__ k_pool,
                                                         const int32_t* __restrict__ block_ids,
                                                         const int32_t* __restrict__ deltas, int n_blocks,
                                                         int num_blocks, int n_kv, int block_size, int ipc,
                                                         const RopeFreq f, int32_t* err) {
  constexpr int H = D / 2;
  constexpr int V = H / 8;                                    // vectors per half row
  constexpr int NI = kRopeNI;
  __shared__ float cs[kRopeMaxBPC][H], sn[kRopeMaxBPC][H];
  __shared__ int tab[kRopeMaxBPC];                           // table of each block slot
  __shared__ int phys_s[kRopeMaxBPC], delta_s[kRopeMaxBPC];
  const int rows = n_kv * block_size;
  const long long ipb = (long long)rows * V;                 // items per block
  const long long i0 = (long long)blockIdx.x * ipc;
  const long long i1 = i0 + ipc < (long long)n_blocks * ipb ? i0 + ipc : (long long)n_blocks * ipb;
  const int b_first = (int)(i0 / ipb);
  const int nb = (int)((i1 - 1) / ipb) - b_first + 1;         // <= kRopeMaxBPC (host sizes ipc)
  const int total = (int)(i1 - i0);
  if (threadIdx.x < nb) {
    const int ph = block_ids[b_first + threadIdx.x], dl = deltas[b_first + threadIdx.x];
    const bool okb = (unsigned)ph < (unsigned)num_blocks;
    if (!okb) set_err(err, PKV_DEV_BAD_BLOCK);
    phys_s[threadIdx.x] = okb ? ph : -1;
    delta_s[threadIdx.x] = dl;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int b = 0; b < nb; ++b) tab[b] = (b > 0 && delta_s[b] == delta_s[b - 1]) ? tab[b - 1] : b;
  }
  const int off0 = (int)(i0 - (long long)b_first * ipb);     // first item's place in block b_first
  uint4 av[NI], bv[NI];
  unsigned live = 0;                                          // bit k: item k of the round is rotated
  // address of the first vector of an item: row r of the block, vector rem % V of its first half
  auto item_ptr = [&](int flat) -> uint4* {
    const int b = flat / (int)ipb, rem = flat - b * (int)ipb, r = rem / V;
    return reinterpret_cast<uint4*>(k_pool + ((size_t)phys_s[b] * rows + r) * D) + (rem - r * V);
  };
  auto load = [&](int base) {
    live = 0;
#pragma unroll
    for (int k = 0; k < NI; ++k) {
      const int idx = base + k * blockDim.x;
      if (idx < total) {
        const int flat = off0 + idx, b = flat / (int)ipb;
        if (phys_s[b] >= 0 && delta_s[b] != 0) {             // else a bad id (flagged) or the identity
          const uint4* p = item_ptr(flat);
          av[k] = p[0];
          bv[k] = p[V];
          live |= 1u << k;
        }
      }
    }
  };
  load(threadIdx.x);
  __syncthreads();                                            // tab
  const double two_pi = 6.283185307179586476925286766559, inv_two_pi = 0.15915494309189533576888376337251;
  for (int e = threadIdx.x; e < nb * H; e += blockDim.x) {
    const int b = e / H, j = e - b * H;
    if (tab[b] != b || delta_s[b] == 0) continue;
    const double ang = (double)delta_s[b] * f.inv_freq[j];
    const double r = fma(-rint(ang * inv_two_pi), two_pi, ang);
    float sv, cv;
    sincosf((float)r, &sv, &cv);
    cs[b][j] = cv;
    sn[b][j] = sv;
  }
  __syncthreads();
  for (int base = threadIdx.x;; base += NI * blockDim.x) {
#pragma unroll
    for (int k = 0; k < NI; ++k) {
      if (!((live >> k) & 1)) continue;
      const int flat = off0 + base + k * blockDim.x;
      const int b = flat / (int)ipb, rem = flat - b * (int)ipb;
      const float* c = cs[tab[b]];
      const float* sr = sn[tab[b]];
      const int j0 = 8 * (rem % V);
      auto rot = [&](uint32_t& wa, uint32_t& wb, int j) {   // channels j, j + 1 and j + H, j + H + 1
        const float x1a = bf16_lo(wa), x1b = bf16_hi(wa), x2a = bf16_lo(wb), x2b = bf16_hi(wb);
        const float y1a = x1a * c[j] - x2a * sr[j], y1b = x1b * c[j + 1] - x2b * sr[j + 1];
        const float y2a = x1a * sr[j] + x2a * c[j], y2b = x1b * sr[j + 1] + x2b * c[j + 1];
        wa = pack_bf16(y1a, y1b);
        wb = pack_bf16(y2a, y2b);
      };
      rot(av[k].x, bv[k].x, j0);
      rot(av[k].y, bv[k].y, j0 + 2);
      rot(av[k].z, bv[k].z, j0 + 4);
      rot(av[k].w, bv[k].w, j0 + 6);
      uint4* p = item_ptr(flat);
      p[0] = av[k];
      p[V] = bv[k];
    }
    if (base + NI * blockDim.x >= total) break;
    load(base + NI * blockDim.x);
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
  // ranges of about 32 KB (1024 items) per CTA: a whole number of blocks, at most
  // kRopeMaxBPC, when blocks are smaller, else 1024 items (then a range touches at most two
  // blocks); 256 threads of kRopeNI items each, fewer for a smaller range
  const long long ipb = (long long)n_kv * block_size * (head_dim / 16);
  long long ipc = 1024;
  if (ipb < 1024) {
    long long k = 1024 / ipb;
    k = k > kRopeMaxBPC ? kRopeMaxBPC : k;
    ipc = k * ipb;
  }
  const long long need = (ipc + kRopeNI - 1) / kRopeNI;
  const int threads = need >= 256 ? 256 : (int)((need + 31) / 32 * 32);
  const long long all = (long long)n_blocks * ipb;
  const unsigned grid = (unsigned)((all + ipc - 1) / ipc);
  if (head_dim == 128)
    rope_shift_kernel<128><<<grid, threads, 0, st>>>(static_cast<__nv_bfloat16*>(k_pool), block_ids, deltas,
                                                     n_blocks, num_blocks, n_kv, block_size, (int)ipc, f, err_flag);
  else
    rope_shift_kernel<64><<<grid, threads, 0, st>>>(static_cast<__nv_bfloat16*>(k_pool), block_ids, deltas,
                                                    n_blocks, num_blocks, n_kv, block_size, (int)ipc, f, err_flag);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    record_cuda_error(e);
    return PKV_ECUDA;
  }
  return PKV_OK;
}
