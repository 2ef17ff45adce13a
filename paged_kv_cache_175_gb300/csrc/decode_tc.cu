// Paged decode attention for groups of 17-32 query heads per kv head (MQA-like layouts) on
// the fifth-generation tensor cores: tcgen05.mma with the accumulators in tensor memory.
//
// Same work partition as the other attention kernels (decode_common.cuh): a persistent CTA
// per SM streams piece p of the (sequence, kv head, block) line.  A tile is up to 128
// tokens -- consecutive blocks of one segment -- and each CTA of 12 warps runs four roles:
//   warps 0, 3   producers: each walks the piece and per tile issues the TMA loads of its K
//                (warp 0) or V (warp 3) blocks (128-byte swizzle, 64-channel boxes) into a
//                ring of 32 KB stages -- 2 for K, freed by the first product, 4 for V, freed
//                by the second -- and warp 0 per segment the group's 32 query rows;
//   warp 1       owner of the tensor memory; one thread issues the first product
//                  S^T[tokens][heads] = K Q^T   (M 128, N 32, K 128; both K-major)
//                into one of two S buffers as soon as a tile's stage has landed;
//   warps 4-11   softmax and epilogue, in two groups of four warps: group g takes heads
//                [16 g, 16 g + 16), and its thread r owns token row r of S^T and channel row
//                r of O^T for those heads (each SM sub-partition runs one role warp and one
//                warp of each group, so the two groups' tiles overlap);
//   warp 2       one thread issues the second product once both groups have written P
//                  O^T[ch][2 x heads] += V^T [P_hi | P_lo]^T
//                                              (M 128, N 64, K = the tile's tokens; V and
//                                               P MN-major, as they lie in shared memory)
//                into one of two O buffers (segment parity).
// Online softmax in base 2 with the scale folded in and a lazy offset (raised only when a
// score exceeds it by more than 8; the raise rescales the O columns in tensor memory and
// each thread's share of the sums l, which the group adds up at the segment's end).  P is
// written to shared memory as a bf16 high part and a bf16 low part (columns 0-31 / 32-63 of
// the second product's B operand), so P's rounding is below 2^-16.
// Rows outside [lead, ntok) and rows of blocks with a bad id get p = 0; their V rows are
// zeroed before the product reads them (a stale row may hold NaN or inf).
#include <cmath>
#include <mutex>

#include "decode_common.cuh"
#include "umma.cuh"

namespace pkv {

struct TcTileMeta {
  int s, g, rows, k;          // rows = ntok | flags << 8 | lead << 16; k = segment number in the piece
  int invalid, nblk, pad0, pad1;
};

template <int BS>
struct TcLayout {
  static constexpr int D = 128;
  static constexpr int TK = 128;                      // tokens per tile
  static constexpr int NBT = TK / BS;                 // blocks per tile
  static constexpr int CHUNK = TK * 128;              // one 64-channel half of K or V: 128 rows x 128 B
  static constexpr int KVST = 2 * CHUNK;              // a K (or V) stage: both halves
  static constexpr int NK = 2, NV = 4;                // K ring and V ring depths
  static constexpr int K_OFF = 0, V_OFF = NK * KVST;
  static constexpr int Q_OFF = V_OFF + NV * KVST;     // 2 query buffers of 2 x (32 rows x 128 B)
  static constexpr int QBUF = 2 * 32 * 128;
  static constexpr int P_OFF = Q_OFF + 2 * QBUF;      // the P buffer: 128 rows x 128 B
  static constexpr int PBUF = TK * 128;
  static constexpr int M_OFF = P_OFF + PBUF;          // metadata, barriers, reduction scratch
  static constexpr int META = (NK + NV) * (int)sizeof(TcTileMeta);
  static constexpr int NBAR = 28;
  static constexpr int RED_OFF = M_OFF + META + NBAR * 8 + 8;
  static constexpr int BYTES = RED_OFF + 256 * 4;
  static constexpr size_t SMEM = 1024 + (size_t)BYTES;  // with the 1024-byte alignment slack
  static_assert(Q_OFF % 1024 == 0 && P_OFF % 1024 == 0, "descriptor alignment");
  static_assert(SMEM <= 232448, "shared memory of one CTA");
  static constexpr uint32_t TMEM_COLS = 256;          // S[2] at 0 / 32, O[2] at 64 / 128
};

// mbarriers: the K ring (full / empty, 2 each), the V ring (4 each), query buffers, S buffers
// (full / read), the P buffer, O buffers, and the final drains of the two issuers
enum : int { BAR_KFULL = 0, BAR_KEMPTY = 2, BAR_VFULL = 4, BAR_VEMPTY = 8, BAR_QFULL = 12, BAR_QEMPTY = 14,
             BAR_SFULL = 16, BAR_SEMPTY = 18, BAR_PFULL = 20, BAR_PEMPTY = 21, BAR_OFULL = 22, BAR_OEMPTY = 24,
             BAR_DRAIN = 26, BAR_DRAIN_PV = 27 };

// 1 / x to within an ulp or two (the normalisation of the output)
__device__ __forceinline__ float rcp_approx(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int BS>
__global__ void __launch_bounds__(384, 1)
    decode_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ CUtensorMap tmq, const DecodeArgs a) {
  using L = TcLayout<BS>;
  constexpr int NBT = L::NBT;
  extern __shared__ uint8_t smem_raw[];
  // aligned by an offset from the array itself, so every access stays a shared-memory one
  uint8_t* sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  TcTileMeta* kmeta = reinterpret_cast<TcTileMeta*>(sm + L::M_OFF);   // per K stage
  TcTileMeta* vmeta = kmeta + L::NK;                                    // per V stage
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + L::M_OFF + L::META);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar + L::NBAR);
  float* red = reinterpret_cast<float*>(sm + L::RED_OFF);          // 256 floats of reduction scratch
  __shared__ volatile int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    abort_flag = 0;
    for (int b = 0; b < L::NBAR; ++b)
      mbar_init(&bar[b], (b == BAR_SEMPTY || b == BAR_SEMPTY + 1 || b == BAR_PFULL || b == BAR_OEMPTY ||
                          b == BAR_OEMPTY + 1) ? 8 : 1);     // one arrival per softmax warp
    fence_barrier_init();
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
    prefetch_tensormap(&tmq);
  }
  if (warp == 1) tmem_alloc(tmem_slot, L::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  if (!a.inline_plan) grid_dep_wait();   // the plan kernel's cum / ctx_eff / cursors
  grid_dep_launch();

  Cursor cur;
  PieceInfo pi;
  piece_setup(a, blockIdx.x, gridDim.x, warp == 0 || warp == 3, cur, pi);   // both producers walk the piece
  const int P = pi.P, p = blockIdx.x;
  const long long pstart = pi.pstart, pend = pi.pend;
  const int len = p < P ? (int)(pend - pstart) : 0;
  // Every thread waits for the kernel before this one (the append) before any read of the
  // pools; the setup above reads only this call's inputs.
  if (warp == 0 && lane == 0 && len > 0) prefetch_l2(a.bt + (size_t)cur.s * a.max_blocks + cur.b0 + cur.blk);
  if (a.inline_plan) grid_dep_wait();

  if (len > 0) {
    if (warp == 0 || warp == 3) {
      // ------------------------------- producers -------------------------------
      // Warp 0 loads K (and, per segment, the group's queries) into a ring of NK stages;
      // warp 3 loads V into a ring of NV stages.  Each walks the same tiles and keeps one tile
      // ahead: the next tile's block ids are fetched while it waits for a free stage, and a
      // tile's copies (2 per block: two 64-channel boxes) go out from one lane each.  K is
      // free again once the first product has run, V only after the second, so the V ring is
      // the deeper one.
      const bool kside = warp == 0;
      const int depth = kside ? L::NK : L::NV;
      const uint64_t pol = policy_evict_first();
      struct Tile {
        int s, g, nblk, rows, k, phys;               // phys: the block id of lane `lane`
      };
      int pj = 0, k = -1, kq = -1;                    // kq: the last segment whose queries were loaded
      auto describe = [&](Tile& t) {
        const bool first = pj == 0 || cur.blk == 0;
        if (first) ++k;
        int nblk = cur.nb - cur.blk;
        nblk = nblk < NBT ? nblk : NBT;
        nblk = nblk < len - pj ? nblk : len - pj;
        const int lb = cur.blk + nblk - 1;                             // the tile's last block
        const bool seg_last = lb == cur.nb - 1, end = pj + nblk >= len;
        const int ntok = (nblk - 1) * BS + (seg_last ? cur.ctx - (cur.b0 + lb) * BS : BS);
        const int lead = cur.blk == 0 ? window_lead(cur.ctx, a.window, BS) : 0;
        int flags = 0;
        if (first) flags |= F_FIRST;
        if (seg_last || end) flags |= F_LAST;
        if (cur.seg_start >= pstart && cur.seg_start + cur.nb <= pend) flags |= F_WHOLE;
        if (end) flags |= F_END;
        const int32_t* row = a.bt + (size_t)cur.s * a.max_blocks + cur.b0;
        t.phys = lane < nblk ? __ldg(row + cur.blk + lane) : -1;
        if (lane == 0 && cur.blk + 2 * NBT < cur.nb) prefetch_l2(row + cur.blk + 2 * NBT);
        t.s = cur.s;
        t.g = cur.g;
        t.nblk = nblk;
        t.rows = pack_rows(ntok, lead, flags);
        t.k = k;
        pj += nblk;
        if (pj < len) {
          cur.blk += nblk - 1;
          cursor_next(cur, a);
        }
      };
      Tile t, tn;
      describe(t);
      int i = 0;
      for (;; ++i) {
        const bool more = pj < len;
        if (more) describe(tn);                                        // its block ids in flight
        const int slot = i % depth, use = i / depth, flags = (t.rows >> 8) & 255, qb = t.k & 1;
        uint64_t* fullb = &bar[(kside ? BAR_KFULL : BAR_VFULL) + slot];
        bool ok = !abort_flag;
        if (ok && i >= depth && lane == 0)
          ok = mbar_wait(&bar[(kside ? BAR_KEMPTY : BAR_VEMPTY) + slot], (use - 1) & 1);
        if (ok && kside && (flags & F_FIRST) && t.k >= 2 && lane == 0)
          ok = mbar_wait(&bar[BAR_QEMPTY + qb], ((t.k >> 1) - 1) & 1);
        ok = __shfl_sync(FULL_MASK, ok, 0);
        if (!ok) {
          if (lane == 0) {
            set_err(a.err, PKV_DEV_TIMEOUT);
            abort_flag = 1;
          }
          break;
        }
        const bool okb = lane < t.nblk && (unsigned)t.phys < (unsigned)a.num_blocks;
        const unsigned invalid = __ballot_sync(FULL_MASK, lane < t.nblk && !okb);
        const unsigned valid = __ballot_sync(FULL_MASK, okb);
        uint8_t* st = sm + (kside ? L::K_OFF + slot * L::KVST : L::V_OFF + slot * L::KVST);
        if (lane == 0) {
          if (invalid && kside) set_err(a.err, PKV_DEV_BAD_BLOCK);
          TcTileMeta mt;
          mt.s = t.s; mt.g = t.g; mt.rows = t.rows; mt.k = t.k;
          mt.invalid = (int)invalid; mt.nblk = t.nblk; mt.pad0 = mt.pad1 = 0;
          (kside ? kmeta : vmeta)[slot] = mt;
          if (kside && (flags & F_FIRST)) {
            uint8_t* qd = sm + L::Q_OFF + qb * L::QBUF;
            const int qrow = t.s * a.n_h + t.g * a.G;
            mbar_arrive_expect_tx(&bar[BAR_QFULL + qb], L::QBUF);
            tma_load_3d(qd, &tmq, 0, qrow, 0, &bar[BAR_QFULL + qb], pol);
            tma_load_3d(qd + L::QBUF / 2, &tmq, 64, qrow, 0, &bar[BAR_QFULL + qb], pol);
            kq = t.k;
          }
          mbar_arrive_expect_tx(fullb, (uint32_t)__popc(valid) * 2u * BS * 128u);
        }
        __syncwarp();
        {
          const int b = lane >> 1, part = lane & 1;                    // lane: block b, box `part`
          const int pb = __shfl_sync(FULL_MASK, t.phys, b & 31);
          if (b < t.nblk && ((valid >> b) & 1))
            tma_load_3d(st + part * L::CHUNK + b * BS * 128, kside ? &tmk : &tmv, part * 64, t.g * BS, pb, fullb,
                        pol);
        }
        if (!more) {
          ++i;
          break;
        }
        t = tn;
      }
      // After a timeout: let the loads already issued land before the CTA leaves (bounded).
      if (abort_flag && lane == 0) {
        bool live = true;
        for (int j = i - depth < 0 ? 0 : i - depth; j < i && live; ++j)
          live = mbar_wait(&bar[(kside ? BAR_KFULL : BAR_VFULL) + j % depth], (j / depth) & 1);
        if (live && kside && kq >= 0) mbar_wait(&bar[BAR_QFULL + (kq & 1)], (kq >> 1) & 1);
      }
      __syncwarp();
    } else if (warp == 1) {
      // ------------------------- first-product issuer -------------------------
      // S^T[i % 2] = K Q^T once tile i's stage and its segment's queries have landed and the
      // softmax has read S buffer i % 2 for tile i - 2.
      if (lane == 0) {
        constexpr uint32_t IQK = umma_idesc_bf16(128, 32, 0, 0);
        const uint32_t sbase = smem_u32(sm);
        bool ok = true;
        for (int i = 0;; ++i) {
          const int slot = i % L::NK, sb = i & 1;
          if (abort_flag || !mbar_wait(&bar[BAR_KFULL + slot], (i / L::NK) & 1)) {
            ok = false;
            break;
          }
          const TcTileMeta mt = kmeta[slot];
          const int flags = (mt.rows >> 8) & 255;
          if (((flags & F_FIRST) && !mbar_wait(&bar[BAR_QFULL + (mt.k & 1)], (mt.k >> 1) & 1)) ||
              (i >= 2 && !mbar_wait(&bar[BAR_SEMPTY + sb], ((i >> 1) - 1) & 1))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t kb = sbase + L::K_OFF + slot * L::KVST, qb = sbase + L::Q_OFF + (mt.k & 1) * L::QBUF;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint64_t ad = umma_desc(kb + (ks >> 2) * L::CHUNK + (ks & 3) * 32, 16, 1024, kLayoutSw128);
            const uint64_t bd = umma_desc(qb + (ks >> 2) * (L::QBUF / 2) + (ks & 3) * 32, 16, 1024, kLayoutSw128);
            umma_bf16(tmem + 32 * sb, ad, bd, IQK, ks > 0 ? 1u : 0u);
          }
          umma_commit(&bar[BAR_SFULL + sb]);
          umma_commit(&bar[BAR_KEMPTY + slot]);
          if (flags & F_LAST) umma_commit(&bar[BAR_QEMPTY + (mt.k & 1)]);
          if (flags & F_END) break;
        }
        if (!ok) {
          set_err(a.err, PKV_DEV_TIMEOUT);
          abort_flag = 1;
        }
        // every product issued has completed before the tensor memory is released
        umma_commit(&bar[BAR_DRAIN]);
        mbar_wait(&bar[BAR_DRAIN], 0);
      }
      __syncwarp();                     // the warp reaches the CTA barrier converged
    } else if (warp == 2) {
      // ------------------------- second-product issuer ------------------------
      // O^T[segment parity] += V^T [P_hi | P_lo]^T once the softmax groups have written tile
      // i's P (and, for a segment's first tile, has read the O buffer's previous segment).
      if (lane == 0) {
        constexpr uint32_t IPV = umma_idesc_bf16(128, 64, 1, 1);
        const uint32_t sbase = smem_u32(sm);
        bool ok = true;
        for (int i = 0;; ++i) {
          const int slot = i % L::NV;
          if (abort_flag || !mbar_wait(&bar[BAR_VFULL + slot], (i / L::NV) & 1) || !mbar_wait(&bar[BAR_PFULL], i & 1)) {
            ok = false;
            break;
          }
          const TcTileMeta mt = vmeta[slot];
          const int flags = (mt.rows >> 8) & 255, ntok = mt.rows & 255, ob = mt.k & 1;
          if ((flags & F_FIRST) && mt.k >= 2 && !mbar_wait(&bar[BAR_OEMPTY + ob], ((mt.k >> 1) - 1) & 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t vb = sbase + L::V_OFF + slot * L::KVST, pb = sbase + L::P_OFF;
          const uint32_t od = tmem + 64 + 64 * ob;
          const int nks = (ntok + 15) >> 4;
          for (int kk = 0; kk < nks; ++kk) {
            const uint64_t ad = umma_desc(vb + kk * 2048, L::CHUNK, 1024, kLayoutSw128);
            const uint64_t bd = umma_desc(pb + kk * 2048, L::CHUNK, 1024, kLayoutSw128);
            const uint32_t acc = ((flags & F_FIRST) && kk == 0) ? 0u : 1u;
            umma_bf16(od, ad, bd, IPV, acc);
          }
          umma_commit(&bar[BAR_VEMPTY + slot]);
          umma_commit(&bar[BAR_PEMPTY]);
          if (flags & F_LAST) umma_commit(&bar[BAR_OFULL + ob]);
          if (flags & F_END) break;
        }
        if (!ok) {
          set_err(a.err, PKV_DEV_TIMEOUT);
          abort_flag = 1;
        }
        umma_commit(&bar[BAR_DRAIN_PV]);
        mbar_wait(&bar[BAR_DRAIN_PV], 0);
      }
      __syncwarp();
    } else {
      // -------------------------- softmax and epilogue ------------------------
      // Group gi of four warps takes heads [hb, hb + 16); warp w reaches the tensor-memory
      // lanes of quarter w % 4, so thread r of a group owns token row r of S^T and channel
      // row r of O^T for its heads.
      const int wq = warp & 3, gi = (warp - 4) >> 2, hb = 16 * gi;
      const int row = 32 * wq + lane;
      const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
      float* redg = red + 64 * gi;                    // [4 warps][16 heads]: the group's maxima
      float* red_m = red + 128;                       // the segment's offsets and sums, 32 heads
      float* red_l = red + 160;
      float m[16], l[16];                             // running offsets (the same in every thread) and
                                                      // this thread's rows' share of the softmax sums
      // A failed (timed-out) wait makes `bad` true for the whole warp; both groups learn of it
      // at the vote that opens each tile and leave together, so no thread is left at a named
      // barrier.  Within a tile every named barrier is passed whatever happened.
      bool bad = false;
      int i = 0;
      for (;;) {
        const int slot = i % L::NV, sb = i & 1;
        bool okw = !bad && !abort_flag && mbar_wait(&bar[BAR_VFULL + slot], (i / L::NV) & 1) &&
                   mbar_wait(&bar[BAR_SFULL + sb], (i >> 1) & 1);
        okw = __all_sync(FULL_MASK, okw);
        if (named_bar_or(1, 256, !okw)) {
          bad = true;
          break;
        }
        const TcTileMeta mt = vmeta[slot];
        const int ntok = mt.rows & 255, flags = (mt.rows >> 8) & 255, lead = mt.rows >> 16, ob = mt.k & 1;
        tc_fence_after();
        float x[16];
        {
          uint32_t sr[16];
          tmem_ld16(tmem + lane_off + 32 * sb + hb, sr);
          tmem_wait_ld();
#pragma unroll
          for (int h = 0; h < 16; ++h) x[h] = __uint_as_float(sr[h]) * a.scale_log2;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bar[BAR_SEMPTY + sb]);     // S buffer sb may be rewritten
        if (flags & F_FIRST) {
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            m[h] = -INFINITY;
            l[h] = 0.f;
          }
        }
        const bool valid = row >= lead && row < ntok && !((mt.invalid >> (row / BS)) & 1);
        bool over = false;
        if (valid) {
#pragma unroll
          for (int h = 0; h < 16; ++h) over |= x[h] > m[h] + kLazyMax;
        } else {
#pragma unroll
          for (int h = 0; h < 16; ++h) x[h] = -INFINITY;
        }
        if (named_bar_or(2 + gi, 128, over)) {
          // raise the group's offsets to the running max.  After the exchange across the two
          // half-warps, a reduce-scatter leaves the warp's max of head hb + (lane & 15) in
          // v[0]; the four warps' maxima meet in shared memory.
          float v[16];
#pragma unroll
          for (int h = 0; h < 16; ++h) v[h] = fmaxf(x[h], __shfl_xor_sync(FULL_MASK, x[h], 16));
#pragma unroll
          for (int o = 8; o >= 1; o >>= 1) {
            const bool up = lane & o;
#pragma unroll
            for (int j = 0; j < o; ++j) {
              const float keep = up ? v[j + o] : v[j], send = up ? v[j] : v[j + o];
              v[j] = fmaxf(keep, __shfl_xor_sync(FULL_MASK, send, o));
            }
          }
          if (lane < 16) redg[wq * 16 + lane] = v[0];
          named_bar(4 + gi, 128);
          const int hl = lane & 15;
          const float mx = fmaxf(fmaxf(redg[hl], redg[16 + hl]), fmaxf(redg[32 + hl], redg[48 + hl]));
          named_bar(4 + gi, 128);
          float al[16];
#pragma unroll
          for (int h = 0; h < 16; ++h) {
            const float mn = fmaxf(m[h], __shfl_sync(FULL_MASK, mx, h));
            al[h] = m[h] == -INFINITY ? 0.f : ex2(m[h] - mn);
            m[h] = mn;
            l[h] *= al[h];
          }
          if (!(flags & F_FIRST)) {
            // O accumulated so far: wait for the previous tile's products, then scale the
            // group's high and low columns in place
            bad |= !__all_sync(FULL_MASK, mbar_wait(&bar[BAR_PEMPTY], (i - 1) & 1));
            if (!bad) {
              tc_fence_after();
#pragma unroll 1
              for (int part = 0; part < 2; ++part) {
                const uint32_t ta = tmem + lane_off + 64 + 64 * ob + 32 * part + hb;
                uint32_t orr[16];
                tmem_ld16(ta, orr);
                tmem_wait_ld();
#pragma unroll
                for (int h = 0; h < 16; ++h) orr[h] = __float_as_uint(__uint_as_float(orr[h]) * al[h]);
                tmem_st16(ta, orr);
                tmem_wait_st();
              }
              tc_fence_before();
            }
          }
        }
        // the P buffer is free once the products of tile i - 1 have completed
        if (i >= 1) bad |= !__all_sync(FULL_MASK, mbar_wait(&bar[BAR_PEMPTY], (i - 1) & 1));
        uint32_t ph[8], pl[8];
#pragma unroll
        for (int h2 = 0; h2 < 8; ++h2) {
          float pv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int h = 2 * h2 + e;
            pv[e] = valid ? ex2(x[h] - m[h]) : 0.f;
            l[h] += pv[e];
          }
          ph[h2] = pack_bf16(pv[0], pv[1]);
          pl[h2] = pack_bf16(pv[0] - bf16_lo(ph[h2]), pv[1] - bf16_hi(ph[h2]));
        }
        // row `row` of the B operand: 128 bytes (high parts of heads 0-31, then low parts),
        // 16-byte chunk c stored at chunk c ^ (row % 8) (128-byte swizzle); this group's
        // heads are chunks 2 gi, 2 gi + 1 (high) and 4 + 2 gi, 5 + 2 gi (low)
        uint8_t* prow = sm + L::P_OFF + row * 128;
        if (!bad) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            *reinterpret_cast<uint4*>(prow + (((2 * gi + c) ^ (row & 7)) << 4)) =
                make_uint4(ph[4 * c], ph[4 * c + 1], ph[4 * c + 2], ph[4 * c + 3]);
            *reinterpret_cast<uint4*>(prow + (((4 + 2 * gi + c) ^ (row & 7)) << 4)) =
                make_uint4(pl[4 * c], pl[4 * c + 1], pl[4 * c + 2], pl[4 * c + 3]);
          }
          if (!valid && row < ((ntok + 15) & ~15)) {      // a V row the product reads with p = 0
            uint8_t* vrow = sm + L::V_OFF + slot * L::KVST + gi * L::CHUNK + row * 128;   // this group's half
#pragma unroll
            for (int c = 0; c < 8; ++c) *reinterpret_cast<uint4*>(vrow + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        fence_proxy_async_smem();          // the rows written above, for the tensor core
        __syncwarp();
        if (lane == 0 && !bad) mbar_arrive(&bar[BAR_PFULL]);

        if (flags & F_LAST) {
          // The segment's softmax sums of the group's heads: a reduce-scatter over the warp
          // leaves the warp's sum of head hb + (lane & 15) in v[0], and the four warps' sums
          // meet in shared memory.  Then O^T of those heads, once the segment's products have
          // completed, and O / l through shared memory (the P buffer, which those products were
          // the last to read) to coalesced stores.
          float ls[16];
          {
            float v[16];
#pragma unroll
            for (int h = 0; h < 16; ++h) v[h] = l[h] + __shfl_xor_sync(FULL_MASK, l[h], 16);
#pragma unroll
            for (int o = 8; o >= 1; o >>= 1) {
              const bool up = lane & o;
#pragma unroll
              for (int j = 0; j < o; ++j) {
                const float keep = up ? v[j + o] : v[j], send = up ? v[j] : v[j + o];
                v[j] = keep + __shfl_xor_sync(FULL_MASK, send, o);
              }
            }
            if (lane < 16) redg[wq * 16 + lane] = v[0];
            named_bar(4 + gi, 128);
            const int hl = lane & 15;
            const float tot = (redg[hl] + redg[16 + hl]) + (redg[32 + hl] + redg[48 + hl]);
            named_bar(4 + gi, 128);
#pragma unroll
            for (int h = 0; h < 16; ++h) ls[h] = __shfl_sync(FULL_MASK, tot, h);
          }
          bad |= !__all_sync(FULL_MASK, !bad && mbar_wait(&bar[BAR_OFULL + ob], (mt.k >> 1) & 1));
          const bool whole = flags & F_WHOLE;
          float* scr = reinterpret_cast<float*>(sm + L::P_OFF);          // [128 channels][32 heads]
          if (!bad) {
            tc_fence_after();
            const uint32_t oc = tmem + lane_off + 64 + 64 * ob + hb;
            uint32_t t0[16], t1[16];
            float o[16];
            tmem_ld16(oc, t0);
            tmem_ld16(oc + 32, t1);
            tmem_wait_ld();
            tc_fence_before();
#pragma unroll
            for (int h = 0; h < 16; ++h) {                              // high part + low part
              o[h] = __uint_as_float(t0[h]) + __uint_as_float(t1[h]);
              if (whole) o[h] *= ls[h] > 0.f ? rcp_approx(ls[h]) : 0.f;
            }
            // row `row`, 4-head group cg at group cg ^ (row % 8): the column reads below then
            // spread over 8 banks
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const int cg = 4 * gi + c;
              *reinterpret_cast<float4*>(scr + row * 32 + 4 * (cg ^ (row & 7))) =
                  make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
            }
            if (!whole && row == 0) {
#pragma unroll
              for (int h = 0; h < 16; ++h) {
                red_m[hb + h] = m[h];
                red_l[hb + h] = ls[h];
              }
            }
          }
          __syncwarp();
          if (lane == 0 && !bad) mbar_arrive(&bar[BAR_OEMPTY + ob]);
          named_bar(6, 256);
          const int tg = threadIdx.x - 128 - 128 * gi;                   // thread of the group
          const int nh = a.G - hb < 16 ? a.G - hb : 16;                  // the group's heads
          if (!bad) {
            const size_t qrow0 = (size_t)mt.s * a.n_h + (size_t)mt.g * a.G + hb;
            const long long part = (long long)mt.s * a.n_kv + mt.g + p;
#pragma unroll 4
            for (int idx = tg; idx < nh * 128; idx += 128) {
              const int hh = idx >> 7, h = hb + hh, c = idx & 127;
              const float v = scr[c * 32 + 4 * ((h >> 2) ^ (c & 7)) + (h & 3)];
              if (!whole) a.ws_o[((size_t)part * a.G + h) * 128 + c] = v;
              else if (a.out_f32) reinterpret_cast<float*>(a.out)[(qrow0 + hh) * 128 + c] = v;
              else reinterpret_cast<__nv_bfloat16*>(a.out)[(qrow0 + hh) * 128 + c] = __float2bfloat16_rn(v);
            }
            if (!whole && tg < nh)
              *reinterpret_cast<float2*>(a.ws_ml + ((size_t)part * a.G + hb + tg) * 2) =
                  make_float2(red_m[hb + tg], red_l[hb + tg]);
          }
          named_bar(6, 256);                 // the scratch is read before the next tile's P lands
        }
        if (flags & F_END) break;
        ++i;
      }
      if (bad && lane == 0) {
        set_err(a.err, PKV_DEV_TIMEOUT);
        abort_flag = 1;
      }
    }
  }
  // the tensor memory is released once every role is done with it (the MMA issuer waited
  // for its last product)
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, L::TMEM_COLS);
}

// ---------------------------------------------------------------------------------------------
template <int BS>
static const void* tc_fn() {
  return (const void*)decode_tc_kernel<BS>;
}

// Kernel and dynamic shared memory of the tensor-memory variant for a block size (head_dim 128).
bool tc_variant(int block_size, const void** fn, size_t* smem) {
  switch (block_size) {
    case 16: *fn = tc_fn<16>(); *smem = TcLayout<16>::SMEM; return true;
    case 32: *fn = tc_fn<32>(); *smem = TcLayout<32>::SMEM; return true;
    case 64: *fn = tc_fn<64>(); *smem = TcLayout<64>::SMEM; return true;
    default: return false;
  }
}

}  // namespace pkv
