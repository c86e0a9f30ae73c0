// bf16 forward of dilution attention on sm_103a tensor cores.
//
// The operator ("DilutionAttention v0.1.0 · results", section "The
// operator") needs every query row's softmax normaliser before any share can
// be formed: share_ik = e_ik / (Z_i (committed_ik + eps) + e_ik) is not
// linear in the normaliser Z_i, so a single online-softmax pass cannot
// produce it.  The forward therefore runs two tensor-core passes over the
// causal triangle plus a memory pass:
//
//  rowstats_kernel  (one CTA per pair of 128-row query tiles)
//     S = Q K^T on tcgen05 (bf16 x bf16 -> fp32 in TMEM), K tiles streamed by
//     TMA through a 4-stage ring; one thread per query row keeps an online
//     max / sum and writes -lse2_i, lse2_i = log2 sum_k 2^(x_ik), x = s * c2,
//     c2 = tau / sqrt(d) * log2(e).  Also zeroes the rows of the fp32
//     accumulator that the sweep adds into.
//
//  sweep_kernel  (one CTA per span of 384 keys, all three tiles resident in smem)
//     Walks the query tiles from the span's diagonal to the end, in causal
//     order.  S^T = K Q^T puts keys on TMEM lanes, so each thread owns one key
//     and carries that key's demand (committed + eps) in a register across
//     query tiles: for each query column in order
//         p = 2^(x - lse2),  den = committed + eps + p,
//         share = p / den,   committed + eps <- den
//     which is exactly the exclusive cumulative sum down the key column.  The
//     shares (bf16) are written to shared memory as the MN-major A operand of
//     a second tcgen05 product, share^T [V | 1]: TMEM columns 0..63 collect
//     sum_k share_ik v_k and columns 64..79 sum_k share_ik (a constant all-ones
//     block).  An epilogue warpgroup adds each query tile's partials into
//     acc[row][0..64] with vector fp32 reductions in L2.  The share^T [V | 1]
//     product is one M = 128, N = 80 instruction per 16 keys.
//
//  finalize (fwd_f32.cu) divides the numerator by the row sum.
//
// Warp specialisation, all waits bounded (timeout -> DA_ERR_TIMEOUT):
//   rowstats: warps 0-3 / 4-7 = softmax-statistics warpgroups for the two
//             query tiles, warp 8 = TMA producer, warp 9 = MMA issuer.
//   sweep:    warps 0-11 = demand warpgroups (key tiles 0..2 of the span),
//             warps 12-15 = epilogue, warp 16 = TMA, warps 17-19 = MMA issuers
//             (one per demand warpgroup).
#include "da_internal.h"
#include "da_ptx.cuh"

#include <cuda.h>
#include <cuda_bf16.h>

namespace da {

// A tile of 128 rows x d bf16 is stored as d / 64 halves of 128 rows x 64
// (128-byte swizzled rows, 16 KB each): 128 bytes is the widest box a
// 128-byte swizzle allows.  Half h of a tile starts h * 16 KB after it.
constexpr uint32_t kHalfBytes = kTile * 64 * 2;
template <int D>
constexpr uint32_t tile_bytes() { return kTile * D * 2; }

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  const uint32_t a = smem_u32(p);
  return p + ((1024u - (a & 1023u)) & 1023u);
}

// Bounded wait that ignores the abort flag: used only to let copies and MMAs
// that are already in flight land before a CTA that gave up exits.
__device__ __forceinline__ void drain_wait(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 100ull * 1000ull * 1000ull) break;
  }
}

// K-major operand tile: 128 rows x 64 bf16 per half (128-byte rows, 128B
// swizzle, as TMA writes it).  8-row groups are 1024 bytes apart; a K step of
// 16 elements advances the start address by 32 bytes inside the swizzle atom,
// and K steps 4.. continue in the next half.
__device__ __forceinline__ uint64_t kmajor_desc(const uint8_t *tile, int kstep) {
  return smem_desc(smem_u32(tile) + (kstep >> 2) * kHalfBytes + (kstep & 3) * 32, 16, 1024);
}

// TMA load of one 128-row tile of a [BH, T, d] tensor into `dst`, half by half.
template <int D>
__device__ __forceinline__ void tma_load_tile(uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int row, int bh) {
#pragma unroll
  for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * kHalfBytes, map, bar, h * 64, row, bh);
}

// After the last tcgen05.ld of a TMEM buffer has completed: hand the buffer
// back to the MMA issuer (one arrival per warp).
__device__ __forceinline__ void release_tmem(uint64_t *bar, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Softmax normaliser of one query row in the log2 domain, lse2 = m + log2 l
// with l = sum 2^(x - m), x = s * c2.  The reference m is the maximum of the
// row's first 32-key chunk (so l >= 1); every later chunk is summed against
// it without a check.  lse2 is exact for any m as long as l stays finite: a
// row whose sum passes 2^120 (a logit more than ~106 above that first
// maximum; fp32 overflows at 2^128) is marked and recomputed exactly by
// rowstats_fixup_kernel.  Terms below 2^-126 flush to zero, which is
// negligible against l >= 1.
struct RowStat {
  float m = -INFINITY;
  float2 l0 = make_float2(0.f, 0.f), l1 = make_float2(0.f, 0.f);

  // 32 consecutive keys (columns col0 ..) of the row; DIAG masks key > query.
  template <bool DIAG>
  __device__ __forceinline__ void chunk(float (&s)[32], int col0, int row, float c2) {
    // every key of the chunk after every row of the warp (6 of the 16
    // warp-chunks of a diagonal tile): nothing to add, exactly as if the
    // masked chunk were summed
    if (DIAG && __all_sync(0xffffffffu, col0 > row)) return;
    if (DIAG) {
#pragma unroll
      for (int c = 0; c < 32; ++c)
        if (col0 + c > row) s[c] = -INFINITY;
    }
    if (m == -INFINITY) {   // the row's first chunk: its maximum becomes the reference
      float t[11];
#pragma unroll
      for (int i = 0; i < 10; ++i) t[i] = fmax3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
      t[10] = fmaxf(s[30], s[31]);
      const float mx =
          fmax3(fmax3(t[0], t[1], t[2]), fmax3(t[3], t[4], t[5]), fmax3(t[6], t[7], fmax3(t[8], t[9], t[10])));
      if (mx == -INFINITY) return;   // every key of the chunk is after the query
      m = mx * c2;
    }
    const float2 c2v = make_float2(c2, c2), nm = make_float2(-m, -m);
#pragma unroll
    for (int j = 0; j < 16; j += 2) {
      const float2 x0 = ffma2(make_float2(s[2 * j], s[2 * j + 1]), c2v, nm);
      const float2 x1 = ffma2(make_float2(s[2 * j + 2], s[2 * j + 3]), c2v, nm);
      l0 = fadd2(l0, make_float2(ex2_approx(x0.x), ex2_approx(x0.y)));
      l1 = fadd2(l1, make_float2(ex2_approx(x1.x), ex2_approx(x1.y)));
    }
  }

  // -lse2 of the row, or NaN when the sum left [1, 2^120] (inf or NaN included).
  __device__ __forceinline__ float neg_lse2() const {
    const float l = (l0.x + l0.y) + (l1.x + l1.y);
    return l <= 0x1p120f ? -(m + log2f(l)) : NAN;
  }
};

// Demand step for 32 consecutive queries (columns 32 C ..) of one key row:
//   p = 2^x,  den = (committed + eps) + p,  share = p / den,
//   committed + eps <- (committed + eps) + p
// (queries in causal order: the exclusive cumsum).  EARLIER (the
// earlier-demand-only variant) takes den = committed + eps instead.
// with x = c2 S' and S' = q.k - lse2 / c2 from the S product (its fifth K
// step adds the -lse2 / c2 term).  MASK zeroes the bids of queries before
// the key: key row `row` is after query column c when row_eff > c,
// row_eff = row - (first query - first key).
template <bool MASK, int C, bool EARLIER>
__device__ __forceinline__ void demand_chunk(const float (&s)[32], int row_eff, float c2, float &ceps,
                                             uint32_t (&pk)[16]) {
  constexpr int col0 = 32 * C;
  const float2 c2v = make_float2(c2, c2);
  float p[32];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const float2 x0 = fmul2(make_float2(s[4 * i], s[4 * i + 1]), c2v);
    const float2 x1 = fmul2(make_float2(s[4 * i + 2], s[4 * i + 3]), c2v);
    p[4 * i] = ex2_approx(x0.x);
    p[4 * i + 1] = ex2_approx(x0.y);
    p[4 * i + 2] = ex2_approx(x1.x);
    p[4 * i + 3] = ex2_approx(x1.y);
  }
  if (MASK) {
#pragma unroll
    for (int c = 0; c < 32; ++c)
      if (row_eff > col0 + c) p[c] = 0.f;
  }
  float d[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) {
    if (EARLIER) {
      d[c] = ceps;
      ceps += p[c];
    } else {
      d[c] = ceps + p[c];
      ceps = d[c];
    }
  }
  // One reciprocal per pair of consecutive queries: r = 1 / (d0 d1),
  // share0 = p0 d1 r, share1 = p1 d0 r.  d0, d1 lie in [eps, T + 1], so
  // d0 d1 stays a normal float for eps >= 1e-18 (and the shares, at most
  // 1 / eps, stay finite).  (Measured on GB300: the
  // MUFU reciprocal of the pair product beats a Newton iteration on the FMA
  // pipe, whose extra instructions cost more issue slots than they save.)
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float r = rcp_approx(d[2 * i] * d[2 * i + 1]);
    const float2 sh = fmul2(fmul2(make_float2(p[2 * i], p[2 * i + 1]), make_float2(d[2 * i + 1], d[2 * i])),
                            make_float2(r, r));
    pk[i] = pack_bf16x2(sh.x, sh.y);
  }
}

// Logit scale of head bh for both kernels.  Masked logits enter as -inf; a
// zero scale (tau = 0) would turn them into NaN, so the scale is at least
// 1e-30, which keeps every finite logit at 0 (uniform bids) and -inf at -inf.
__device__ __forceinline__ float bf16_c2(const HeadScale &hs, int bh, int *status) {
  return fmaxf(head_c2(hs, bh, status), 1e-30f);
}

// ============================================================================
// Row statistics
// ============================================================================
// d = 64: 2 CTAs per SM, one S buffer per query tile (256 TMEM columns);
// d = 128: the tiles take one SM's shared memory, so one CTA per SM with two
// S buffers per query tile (512 columns) keeps the tensor pipe busy while a
// buffer is being reduced.
constexpr int kRsThreads = 320;
constexpr int kRsKStages = 4;
template <int D>
struct RsCfg {
  static constexpr uint32_t kTB = tile_bytes<D>();
  static constexpr int kSlots = D == 64 ? 1 : 2;     // S buffers per query tile
  static constexpr int kCtasPerSm = D == 64 ? 2 : 1;
  static constexpr uint32_t kTmemCols = 2 * kSlots * kTile;
  static constexpr int kSmemBytes = (2 + kRsKStages) * kTB + 256 + 1024;
};

template <int D>
__global__ void __launch_bounds__(kRsThreads, RsCfg<D>::kCtasPerSm)
    rowstats_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    float *__restrict__ nlse2, float *__restrict__ acc, int BH, int T, int Tp, HeadScale hs,
                    int *status) {
  using C = RsCfg<D>;
  constexpr uint32_t kTB = C::kTB;
  constexpr int NS = C::kSlots;
  constexpr int AS = acc_stride(D);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sQ = smem;                    // 2 query tiles
  uint8_t *sK = smem + 2 * kTB;          // K ring
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (2 + kRsKStages) * kTB);
  uint64_t *q_full = bars;
  uint64_t *k_full = bars + 1;
  uint64_t *k_empty = k_full + kRsKStages;
  uint64_t *s_full = k_empty + kRsKStages;   // [g * NS + slot]
  uint64_t *s_free = s_full + 2 * NS;
  uint64_t *drain = s_free + 2 * NS;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const TileWork w = rowstats_work(blockIdx.x, BH, T, D);
  const int n_kt = w.q_tile0 + 2;   // key tiles 0 .. last query tile
  const float c2 = bf16_c2(hs, w.bh, status);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kRsKStages; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
    }
    for (int g = 0; g < 2 * NS; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&s_free[g], 4);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, status};

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmK);
      mbar_arrive_expect_tx(q_full, 2 * kTB);
      tma_load_tile<D>(sQ, &tmQ, q_full, w.q_tile0 * kTile, w.bh);
      tma_load_tile<D>(sQ + kTB, &tmQ, q_full, (w.q_tile0 + 1) * kTile, w.bh);
      int issued = 0;
      for (int kt = 0; kt < n_kt; ++kt) {
        const int s = kt % kRsKStages;
        if (!mbar_wait(&k_empty[s], ((kt / kRsKStages) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(&k_full[s], kTB);
        tma_load_tile<D>(sK + s * kTB, &tmK, &k_full[s], kt * kTile, w.bh);
        ++issued;
      }
      if (*abort_flag) {
        drain_wait(q_full, 0);
        for (int kt = (issued > kRsKStages ? issued - kRsKStages : 0); kt < issued; ++kt)
          drain_wait(&k_full[kt % kRsKStages], (kt / kRsKStages) & 1);
      }
    }
  } else if (warp == 9) {
    // ----------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kTile, kTile, false, false);
      const uint64_t dQ0 = kmajor_desc(sQ, 0), dQ1 = kmajor_desc(sQ + kTB, 0), dK0 = kmajor_desc(sK, 0);
      auto kt_slot = [](int g, int kt) { return g * NS + kt % NS; };
      // d = 64 (two CTAs per SM, four reduction warps per sub-partition):
      // key tile by key tile, query tile 0 then 1, with blocking waits that
      // leave the issue slots to the reduction warps (polling both slots, as
      // at d = 128, measured 0.958 -> 0.989 ms here).
      if (D == 64 && mbar_wait(q_full, 0, wc)) {
        tc_fence_after();
        for (int kt = 0; kt < n_kt; ++kt) {
          const int s = kt % kRsKStages;
          if (!mbar_wait(&k_full[s], (kt / kRsKStages) & 1, wc)) break;
          tc_fence_after();
          bool ok = true;
          for (int g = 0; g < 2; ++g) {
            if (kt > w.q_tile0 + g) continue;   // key tile entirely after this query tile
            // key tile kt is use kt / NS of slot kt % NS of query tile g
            const int slot = g * NS + kt % NS;
            if (!mbar_wait(&s_free[slot], ((kt / NS) & 1) ^ 1, wc)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d = tmem + slot * kTile;
            const uint64_t dQg = g ? dQ1 : dQ0;
            const uint64_t dKs = dK0 + (uint64_t)s * (kTB >> 4);
            MmaRun<0, 4, 2, 2, false>::go(d, dQg, dKs, idesc, 0u);
            if constexpr (D == 128) MmaRun<0, 4, 2, 2, false>::go(d, dQg + (kHalfBytes >> 4), dKs + (kHalfBytes >> 4), idesc, 1u);
            mma_commit(&s_full[slot]);
          }
          if (!ok) break;
          mma_commit(&k_empty[s]);
        }
      }
      // d = 128 (one CTA per SM, two reduction warps per sub-partition): the
      // two query tiles' S products are issued as soon as each one's slot is
      // free, whichever comes first, so that neither tile's reduction waits
      // on the other's (measured: 1.43 -> 1.38 ms at 4x12x16384x128).  Query tile g uses key tiles 0 .. q_tile0 + g;
      // a key stage goes back to the producer once every query tile that uses
      // it has been issued (the commit covers all earlier products).  A query
      // tile runs at most one ring's depth ahead of the other, so no barrier
      // is polled more than one phase ahead.
      if (D == 128 && mbar_wait(q_full, 0, wc)) {
        tc_fence_after();
        const int lim[2] = {w.q_tile0 + 1, w.q_tile0 + 2};
        int nx[2] = {0, 0}, kdone = 0;
        unsigned long long idle0 = 0;
        while (nx[0] < lim[0] || nx[1] < lim[1]) {
          bool progressed = false;
#pragma unroll
          for (int g = 0; g < 2; ++g) {
            const int kt = nx[g];
            if (kt >= lim[g]) continue;
            const int s = kt % kRsKStages;
            const int slot = g * NS + kt % NS;
            if (!mbar_test_wait(&k_full[s], (kt / kRsKStages) & 1) ||
                !mbar_test_wait(&s_free[slot], ((kt / NS) & 1) ^ 1))
              continue;
            tc_fence_after();
            const uint32_t d = tmem + slot * kTile;
            const uint64_t dQg = g ? dQ1 : dQ0;
            const uint64_t dKs = dK0 + (uint64_t)s * (kTB >> 4);
            MmaRun<0, 4, 2, 2, false>::go(d, dQg, dKs, idesc, 0u);
            if constexpr (D == 128) MmaRun<0, 4, 2, 2, false>::go(d, dQg + (kHalfBytes >> 4), dKs + (kHalfBytes >> 4), idesc, 1u);
            mma_commit(&s_full[slot]);
            ++nx[g];
            progressed = true;
          }
          while (kdone < n_kt && (nx[0] > kdone || kdone >= lim[0]) && nx[1] > kdone) {
            mma_commit(&k_empty[kdone % kRsKStages]);
            ++kdone;
          }
          if (progressed) {
            idle0 = 0;
            continue;
          }
          if (*abort_flag) break;
          const unsigned long long now = globaltimer();
          if (idle0 == 0) {
            idle0 = now;
          } else if (now - idle0 > kWaitLimitNs) {
            raise_timeout(wc, nx[0] < lim[0] ? &s_free[kt_slot(0, nx[0])] : &s_free[kt_slot(1, nx[1])]);
            break;
          }
          __nanosleep(32);
        }
      }
      mma_commit(drain);
      drain_wait(drain, 0);
    }
  } else {
    // ------------------------------------------- softmax statistics (2 WGs)
    const int g = warp / 4;
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;
    const int qt = w.q_tile0 + g;
    const int64_t qi = (int64_t)qt * kTile + row;
    RowStat st;
    for (int kt = 0; kt <= qt; ++kt) {
      const int slot = g * NS + kt % NS;
      const uint32_t tbase = tmem + slot * kTile + ((uint32_t)(quarter * 32) << 16);
      if (!warp_wait(&s_full[slot], (kt / NS) & 1, wc)) break;
      tc_fence_after();
      // 32-column chunks; the load of chunk c+1 is in flight while chunk c is reduced.
      float A[32], B[32];
      if (kt < qt) {
        tmem_ld32(tbase, A);
        tmem_wait_ld_r(A);
        tmem_ld32(tbase + 32, B);
        st.chunk<false>(A, 0, row, c2);
        tmem_wait_ld_r(B);
        tmem_ld32(tbase + 64, A);
        st.chunk<false>(B, 32, row, c2);
        tmem_wait_ld_r(A);
        tmem_ld32(tbase + 96, B);
        st.chunk<false>(A, 64, row, c2);
        tmem_wait_ld_r(B);
        release_tmem(&s_free[slot], lane);
        st.chunk<false>(B, 96, row, c2);
      } else {
        tmem_ld32(tbase, A);
        tmem_wait_ld_r(A);
        tmem_ld32(tbase + 32, B);
        st.chunk<true>(A, 0, row, c2);
        tmem_wait_ld_r(B);
        tmem_ld32(tbase + 64, A);
        st.chunk<true>(B, 32, row, c2);
        tmem_wait_ld_r(A);
        tmem_ld32(tbase + 96, B);
        st.chunk<true>(A, 64, row, c2);
        tmem_wait_ld_r(B);
        release_tmem(&s_free[slot], lane);
        st.chunk<true>(B, 96, row, c2);
      }
      if (*abort_flag) break;
    }
    if (qi < Tp) {
      // negated, so the sweep forms x - lse2 with one packed fma
      float v = -INFINITY;
      if (qi < T) {
        v = st.neg_lse2();
        if (v != v) atomicAdd(status + kStatusRowsRedo, 1);   // marked for rowstats_fixup_kernel
      }
      nlse2[(size_t)w.bh * Tp + qi] = v;
      float4 *ar = reinterpret_cast<float4 *>(acc + ((size_t)w.bh * Tp + qi) * AS);
#pragma unroll
      for (int t = 0; t < AS / 4; ++t) ar[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// Exact recomputation of the rows that rowstats_kernel marked (their running
// sum overflowed: a logit more than ~106 above the maximum of the row's first
// 32 keys).  One warp per marked row: each lane walks keys lane, lane + 32, ...
// <= the query with an exact running maximum, then the lanes' (max, sum)
// pairs are merged.  Exits at once when no row was marked, which is the case
// for any input whose logits stay within ~106 (log2 units) of each row's
// first-chunk maximum.
template <int D>
__global__ void __launch_bounds__(256) rowstats_fixup_kernel(const __nv_bfloat16 *__restrict__ q,
                                                             const __nv_bfloat16 *__restrict__ k,
                                                             float *__restrict__ nlse2, int BH, int T, int Tp,
                                                             HeadScale hs, int *status) {
  // nothing marked, or the pass gave up (rows it did not reach are not valid marks)
  const volatile int *vs = status;
  if (vs[kStatusRowsRedo] == 0 || vs[0] != DA_OK) return;
  __shared__ float sq[8][D];
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int64_t nrows = (int64_t)BH * Tp;
  const int64_t nwarps = (int64_t)gridDim.x * 8;
  for (int64_t base = ((int64_t)blockIdx.x * 8 + warp) * 32; base < nrows; base += nwarps * 32) {
    const bool marked = base + lane < nrows && nlse2[base + lane] != nlse2[base + lane];
    uint32_t todo = __ballot_sync(0xffffffffu, marked);
    while (todo != 0u) {
      const int64_t r = base + (__ffs(todo) - 1);
      todo &= todo - 1u;
      const int bh = (int)(r / Tp);
      const int64_t i = r % Tp;
      if (i >= T) continue;       // padded rows are never marked
      const float c2 = bf16_c2(hs, bh, nullptr);
      for (int t = lane; t < D; t += 32) sq[warp][t] = __bfloat162float(q[((size_t)bh * T + i) * D + t]);
      __syncwarp();
      float m = -INFINITY, l = 0.f;
      for (int64_t key = lane; key <= i; key += 32) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(k + ((size_t)bh * T + key) * D);
        float dot = 0.f;
#pragma unroll
        for (int t = 0; t < D / 8; ++t) {
          const uint4 u = __ldg(kr + t);
          const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&w4[e]));
            dot = fmaf(sq[warp][8 * t + 2 * e], kv.x, dot);
            dot = fmaf(sq[warp][8 * t + 2 * e + 1], kv.y, dot);
          }
        }
        const float x = dot * c2;
        if (x > m) {
          l = l * ex2_approx(m - x) + 1.f;
          m = x;
        } else {
          l += ex2_approx(x - m);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float mo = __shfl_xor_sync(0xffffffffu, m, o), lo = __shfl_xor_sync(0xffffffffu, l, o);
        const float mn = fmaxf(m, mo);
        l = (mn == -INFINITY) ? 0.f : l * ex2_approx(m - mn) + lo * ex2_approx(mo - mn);
        m = mn;
      }
      if (lane == 0) nlse2[r] = -(m + log2f(l));
      __syncwarp();
    }
  }
}

// ============================================================================
// Demand sweep
// ============================================================================
// One CTA per span of 384 keys (three 128-key tiles, resident with their
// values).  For each 128-query tile, in causal order:
//   S^T_g = K_g Q^T (M = 128 keys, N = 128 queries) into TMEM slot g;
//   demand warpgroup g turns its slot into shares (bf16, shared memory) = the
//   MN-major A operand of D[q, 0:80] += share^T [V_g | 1] (M = 128 queries,
//   N = 80: the value tile and, through the descriptor's leading-byte offset,
//   a 2 KB block of ones whose product is the share row sum); the epilogue
//   adds D into acc[row][0..64].
// Every tcgen05.mma costs at least ~46 cycles on this part and reaches full
// rate only at M = 128, N >= 128, which is why the query tile is 128 wide and
// the row sum rides in the same instruction as the value product.
constexpr int kSwBQ = kSweepQTile;              // 128 queries per tile
constexpr uint32_t kShBytes = 2 * 16 * 1024;    // share^T: 2 M-blocks x 16 key groups x 1 KB
constexpr uint32_t kStageBytes = 32 * 32 * 4;   // epilogue reduction box: 32 rows x 32 fp32, 128B-swizzled
constexpr uint32_t kExtBytes = 128 * 16 * 2;    // one 128-row x 16 bf16 K-major operand, no swizzle
// Register split across warpgroups (setmaxnreg).  The block is launched with
// its threads x (registers per thread) registers; the split must not exceed
// that (checked on the host before every launch).
constexpr int kSwRegsDemand = 128, kSwRegsEpi = 56;

// Per-head-dimension layout.  d = 64: three demand warpgroups (384-key
// spans).  d = 128: two (256-key spans), so that the S slots, the
// accumulators and key tile 0 fit the 512 TMEM columns and the tiles fit
// 227 KB of shared memory; its value product is split into D[q, 0:80] +=
// share^T [V_lo | 1] and DHi[q, 0:64] += share^T V_hi.
template <int D>
struct SwCfg {
  static constexpr int kG = D == 64 ? 3 : 2;           // demand warpgroups, one per key tile
  static constexpr int kWarps = (kG + 2) * 4;         // demand WGs, epilogue WG, producer/MMA WG
  static constexpr int kThreads = kWarps * 32;        // 640 / 512
  static constexpr uint32_t kTB = tile_bytes<D>();
  // control warps: 40 registers at d = 64; the d = 128 issuers keep two more
  // operand descriptors live
  static constexpr int kRegsCtl = D == 64 ? 40 : 56;
  // registers per thread at launch (d = 64: 640 threads leave 96)
  static constexpr int kRegsLaunch = D == 64 ? 96 : 112;
  static constexpr int kRegsNeeded = 128 * (kG * kSwRegsDemand + kSwRegsEpi + kRegsCtl);
  static constexpr uint32_t kOffK = 0;                              // key tiles 1.. (tile 0 is in TMEM)
  static constexpr uint32_t kOffV = kOffK + (kG - 1) * kTB;
  static constexpr uint32_t kOffQ = kOffV + kG * kTB;               // the query tile
  static constexpr uint32_t kOffAExt = kOffQ + kTB;                 // [1 1 1 0 ..] for every key
  static constexpr uint32_t kOffBExt = kOffAExt + kExtBytes;        // [hi mid lo 0 ..] of -lse2 / c2 per query
  static constexpr uint32_t kOffSh = D == 64 ? kOffQ + 2 * kTB : kOffBExt + kExtBytes;
  static constexpr uint32_t kOffOnes = kOffSh + kG * kShBytes;      // above every V tile (positive LBO)
  static constexpr uint32_t kOffStage = kOffOnes + 2048;            // one box per epilogue warp
  static constexpr uint32_t kOffBar = kOffStage + 4 * kStageBytes;
  static constexpr int kSmemBytes = kOffBar + 512;   // the dynamic shared-memory base is 1024-byte aligned
  // TMEM: S^T slots at g * 128; D (80 columns: values 0..63, row sum at 64);
  // DHi (d = 128: values 64..127); key tile 0 as the A operand of its S
  // product (one key per lane, d / 2 columns of bf16 pairs).
  static constexpr uint32_t kTmemD = kG * kTile;
  static constexpr uint32_t kTmemDHi = kTmemD + 80;
  static constexpr uint32_t kTmemK0 = kTmemDHi + (D - 64);
  static_assert(kSmemBytes <= 232448, "sweep shared memory");
  static_assert(kOffStage % 1024 == 0, "reduction boxes are 128B-swizzled");
  static_assert(kRegsNeeded <= 65536, "sweep register split");
  static_assert(kOffBExt + kExtBytes <= kOffSh, "extension operands");
  static_assert(kTmemK0 + D / 2 <= 512, "TMEM columns");
};

__device__ __forceinline__ void regs_inc_demand() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSwRegsDemand)); }
__device__ __forceinline__ void regs_dec_epi() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kSwRegsEpi)); }
template <int N>
__device__ __forceinline__ void regs_dec_ctl() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }

// CHK: also write the demand checkpoints (the backward's forward-again pass).
template <int D, bool EARLIER, bool CHK>
__global__ void __launch_bounds__(SwCfg<D>::kThreads, 1) __maxnreg__(SwCfg<D>::kRegsLaunch)
    sweep_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmAcc,
                 const uint4 *__restrict__ kglob, const float *__restrict__ nlse2, float *__restrict__ acc,
                 float *__restrict__ demand_out, float *__restrict__ cchk, int BH,
                 int T, int Tp, HeadScale hs, float eps, int *status) {
  using C = SwCfg<D>;
  constexpr int kG = C::kG;
  constexpr uint32_t kTB = C::kTB;
  constexpr int AS = acc_stride(D);
  extern __shared__ __align__(1024) uint8_t sw_smem_raw[];
  // The layout has no slack for re-alignment: every tile, swizzle atom and
  // reduction box assumes a 1024-byte aligned base.  Refuse (uniformly,
  // before any barrier) rather than compute with misaligned operands.
  if (smem_u32(sw_smem_raw) & 1023u) {
    if (threadIdx.x == 0) atomicCAS(status, DA_OK, DA_ERR_UNSUPPORTED);
    return;
  }
  uint8_t *smem = sw_smem_raw;
  uint8_t *sK = smem + C::kOffK;
  uint8_t *sV = smem + C::kOffV;
  uint8_t *sQ = smem + C::kOffQ;
  uint8_t *sSh = smem + C::kOffSh;
  uint8_t *sAExt = smem + C::kOffAExt;
  uint8_t *sBExt = smem + C::kOffBExt;
  uint8_t *sOnes = smem + C::kOffOnes;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *kv_full = bars;
  uint64_t *k0_full = kv_full + 1;             // key tile 0 written to TMEM
  uint64_t *q_full = k0_full + 1;              // query tile and its -lse2 / c2 block loaded
  uint64_t *q_empty = q_full + 1;              // every S product of the tile completed
  uint64_t *s_full = q_empty + 1;              // [g]
  uint64_t *s_free = s_full + kG;            // [g]
  uint64_t *sh_full = s_free + kG;           // [g]
  uint64_t *sh_free = sh_full + kG;          // [g]
  uint64_t *d_full = sh_free + kG;
  uint64_t *d_free = d_full + 1;
  uint64_t *drain = d_free + 1;                // [g]: per issuer
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + kG);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int wg = warp / 4;
  const int kWarpProd = (kG + 1) * 4, kWarpMma = kWarpProd + 1;
  const TileWork w = sweep_work(blockIdx.x, BH, T, D);
  const int nt = w.n_q_tiles;
  const float c2 = bf16_c2(hs, w.bh, nullptr);   // the row statistics report bad entries

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    mbar_init(k0_full, 4);
    mbar_init(q_full, 2);      // the tile's bytes + the producer's -lse2 / c2 block
    mbar_init(q_empty, kG);  // one commit per issuer
    for (int g = 0; g < kG; ++g) {
      mbar_init(&s_full[g], 1);
      mbar_init(&s_free[g], 4);
      mbar_init(&sh_full[g], 4);
      mbar_init(&sh_free[g], 1);
    }
    mbar_init(d_full, kG);   // one commit per issuer
    mbar_init(d_free, 4);      // phase t: D holds zeros for tile t (the epilogue warps)
    for (int g = 0; g < kG; ++g) mbar_init(&drain[g], 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  // Constant all-ones block: the N = 64..79 part of the value operand.
  for (int e = threadIdx.x; e < 2048 / 4; e += C::kThreads) reinterpret_cast<uint32_t *>(sOnes)[e] = 0x3F803F80u;
  // The fifth K step of S: A_ext rows (every key) = [1 1 1 0 ... 0], B_ext rows
  // (every query) = [hi mid lo 0 ... 0] of -lse2 / c2 (written per tile), so
  // S' = q.k - lse2 / c2 and x = c2 S'.  K-major, no swizzle: 8-row groups of
  // 256 bytes, each the core matrix of K 0..7 followed by that of K 8..15.
  for (int e = threadIdx.x; e < (int)(kExtBytes / 16); e += C::kThreads) {
    const bool k_lo = (e & 15) < 8;
    reinterpret_cast<uint4 *>(sAExt)[e] = k_lo ? make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
    reinterpret_cast<uint4 *>(sBExt)[e] = make_uint4(0u, 0u, 0u, 0u);
  }
  fence_proxy_async_smem();
  if (warp == kWarpMma) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, status};

  if (wg == kG + 1) {
    regs_dec_ctl<C::kRegsCtl>();
    if (warp == kWarpProd) {
      // ---------------------------------------------------------- producer
      // Lane 0 issues the TMA loads; once the S products of the previous tile
      // (which read both the query tile and B_ext) are done, the 32 lanes turn
      // the tile's -lse2 into B_ext rows, four queries each.
      if (lane == 0) {
        prefetch_tmap(&tmQ);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        prefetch_tmap(&tmAcc);
        mbar_arrive_expect_tx(kv_full, (2 * kG - 1) * kTB);
        for (int g = 0; g < kG; ++g) {
          if (g > 0) tma_load_tile<D>(sK + (g - 1) * kTB, &tmK, kv_full, w.key0 + g * kTile, w.bh);
          tma_load_tile<D>(sV + g * kTB, &tmV, kv_full, w.key0 + g * kTile, w.bh);
        }
      }
      const float4 *lsrc = reinterpret_cast<const float4 *>(nlse2 + (size_t)w.bh * Tp) + lane;
      int q_issued = 0;
      for (int t = 0; t < nt; ++t) {
        const int qrow = (w.q_tile0 + t) * kSwBQ;
        const float4 nl = __ldg(lsrc + qrow / 4);   // -lse2 of queries qrow + 4 lane .. + 3 (-inf past T)
        if (!warp_wait(q_empty, (t & 1) ^ 1, wc)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(q_full, kTB);
          tma_load_tile<D>(sQ, &tmQ, q_full, qrow, w.bh);
        }
        ++q_issued;
        const float nv[4] = {nl.x, nl.y, nl.z, nl.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // -lse2 / c2 as hi + mid + lo bf16 parts (24 significant bits).  Rows
          // past T get a large finite negative value: their bids vanish, and
          // the zero K columns of A_ext that meet it stay 0.
          const float v = fmaxf(nv[j] / c2, -3.0e38f);
          const __nv_bfloat16 h = __float2bfloat16_rn(v);
          const float r1 = v - __bfloat162float(h);
          const __nv_bfloat16 m = __float2bfloat16_rn(r1);
          const __nv_bfloat16 l = __float2bfloat16_rn(r1 - __bfloat162float(m));
          const int q = 4 * lane + j;
          *reinterpret_cast<uint4 *>(sBExt + (q >> 3) * 256 + (q & 7) * 16) =
              make_uint4((uint32_t)__bfloat16_as_ushort(h) | ((uint32_t)__bfloat16_as_ushort(m) << 16),
                         (uint32_t)__bfloat16_as_ushort(l), 0u, 0u);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);
      }
      if (lane == 0 && *abort_flag) {
        drain_wait(kv_full, 0);
        if (q_issued > 0) drain_wait(q_full, (q_issued - 1) & 1);
      }
    } else if (warp >= kWarpMma && warp < kWarpMma + kG && lane == 0) {
      // ------------------------------------------------------- MMA issuers
      // One issuing thread per demand warpgroup (warps 17, 18, 19: one per
      // sub-partition 1..3), each issuing its warpgroup's S and share.[V|1]
      // products.  A tcgen05.mma issue stream slows to a fraction when other
      // warps of its sub-partition are busy, and every sub-partition hosts
      // three demand warps: three streams keep the tensor pipe fed.  All PV
      // products accumulate into D (the epilogue zeroes it after each drain),
      // so their order across issuers does not matter; a commit tracks only
      // its own thread's MMAs, hence q_empty and d_full count one arrival per
      // issuer.
      //   S(t)[g] reads query slot t % 2 (reloaded once all S(t) completed);
      //   PV(t)[g] waits until D holds zeros for tile t (d_free phase t).
      //   Operand descriptors are built once; a K step advances them by a
      //   constant inside the issue sequence (MmaRun): K-major tiles +32 bytes
      //   (+2 in the start field); share^T +2048 bytes (+128); [V | 1] start
      //   +128 and its leading byte offset to the ones block -128 (field at
      //   bit 16).
      const int g = warp - kWarpMma;
      constexpr long long kStepKm = 2, kStepSh = 128, kStepV = 128 - (128ll << 16);
      constexpr uint64_t kTileStep = kTB >> 4, kShStep = kShBytes >> 4;
      constexpr uint64_t kVTileStep = kTileStep - (kTileStep << 16);
      const uint32_t idesc_s = idesc_bf16(kTile, kSwBQ, false, false);
      const uint32_t idesc_pv = idesc_bf16(kSwBQ, 64 + 16, true, true);
      const uint32_t idesc_pv_hi = idesc_bf16(kSwBQ, 64, true, true);   // d = 128: value columns 64..127
      const uint32_t ones_addr = smem_u32(sOnes);
      const uint64_t dQ = kmajor_desc(sQ, 0);
      // fifth K step: -lse2 / c2 for every (key, query)
      const uint64_t dAExt = smem_desc_noswizzle(smem_u32(sAExt), 128, 256);
      const uint64_t dBExt = smem_desc_noswizzle(smem_u32(sBExt), 128, 256);
      const uint64_t dKg = kmajor_desc(sK + (g > 0 ? g - 1 : 0) * kTB, 0);   // (tile 0 is read from TMEM)
      const uint64_t dShg = smem_desc(smem_u32(sSh), 16384, 1024) + g * kShStep;
      const uint64_t dVg = smem_desc(smem_u32(sV), ones_addr - smem_u32(sV), 1024) + g * kVTileStep;
      // d = 128: the value tile's second half (columns 64..127), one N block.
      const uint64_t dVg_hi = smem_desc(smem_u32(sV) + kHalfBytes, kHalfBytes, 1024) + g * kTileStep;
      // Per warpgroup the events come in a fixed order: S(t+1) becomes ready
      // (slot released while tile t is read) before PV(t) (its shares
      // written), so the issuer walks S(0), S(1), PV(0), S(2), PV(1), ... with
      // blocking waits, during which it sleeps instead of taking issue slots
      // from the demand warps of its sub-partition.
      bool ok = mbar_wait(kv_full, 0, wc) && (g != 0 || mbar_wait(k0_full, 0, wc));
      if (ok) tc_fence_after();
      for (int t = 0; ok && t <= nt; ++t) {
        if (t < nt) {
          // S(t)[g] = K_g Q(t)^T into slot g
          if (!mbar_wait(q_full, t & 1, wc) || !mbar_wait(&s_free[g], (t & 1) ^ 1, wc)) break;
          tc_fence_after();
          // K steps 0..3 read the first 64 columns of Q and K, steps 4..7
          // (d = 128) the second halves, 16 KB on (8 TMEM columns per step
          // for key tile 0, which sits in TMEM).
          constexpr long long kHalfStep = kHalfBytes >> 4;
          if (g == 0) {
            MmaRun<0, 4, 8, kStepKm, true>::go(tmem, tmem + C::kTmemK0, dQ, idesc_s, 0u);
            if constexpr (D == 128)
              MmaRun<0, 4, 8, kStepKm, true>::go(tmem, tmem + C::kTmemK0 + 32, dQ + kHalfStep, idesc_s, 1u);
          } else {
            MmaRun<0, 4, kStepKm, kStepKm, false>::go(tmem + g * kTile, dKg, dQ, idesc_s, 0u);
            if constexpr (D == 128)
              MmaRun<0, 4, kStepKm, kStepKm, false>::go(tmem + g * kTile, dKg + kHalfStep, dQ + kHalfStep, idesc_s,
                                                       1u);
          }
          mma_bf16_at<0, 0>(tmem + g * kTile, dAExt, dBExt, idesc_s, 1u);
          mma_commit(&s_full[g]);
          mma_commit(q_empty);
        }
        if (t >= 1) {
          // PV(t-1)[g]: D += share^T [V_g | 1] once D holds zeros for tile t-1
          const int tp = t - 1;
          if (!mbar_wait(d_free, tp & 1, wc) || !mbar_wait(&sh_full[g], tp & 1, wc)) break;
          tc_fence_after();
          // share^T: MN-major, 64-query blocks 16 KB apart (LBO), 8-key groups 1 KB apart (SBO).
          // [V | 1]: MN-major; N block 0 = the value tile's 16 key rows, N block 1 (LBO
          // away) = the ones block, of which N = 64..79 are read.
          MmaRun<0, kTile / 16, kStepSh, kStepV, false>::go(tmem + C::kTmemD, dShg, dVg, idesc_pv, 1u);
          if constexpr (D == 128)
            MmaRun<0, kTile / 16, kStepSh, 128, false>::go(tmem + C::kTmemDHi, dShg, dVg_hi, idesc_pv_hi, 1u);
          mma_commit(&sh_free[g]);
          mma_commit(d_full);
        }
      }
      mma_commit(&drain[g]);
      drain_wait(&drain[g], 0);
    }
  } else if (wg == kG) {
    // -------------------------------------------------------------- epilogue
    // D -> acc through the copy engine: each warp stages its 32 rows x 32
    // columns as a 128B-swizzled box and issues a TMA add-reduction into acc
    // (d / 32 boxes per tile: D's value columns, then DHi's at d = 128); the
    // row sum (D column 64, acc column d) goes by one atomic per row.
    regs_dec_epi();
    const int quarter = warp % 4;
    uint8_t *stage = smem + C::kOffStage + quarter * kStageBytes;
    uint8_t *srow = stage + lane * 128;
    const int swz = lane & 7;
    auto stage_box = [&](const float (&x)[32], int col0, int grow0) {
      if (lane == 0) bulk_wait_read_all();   // the previous box has been read
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<float4 *>(srow + ((j ^ swz) << 4)) =
            make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        tma_reduce_add_2d(&tmAcc, stage, col0, grow0);
        bulk_commit_group();
      }
    };
    // D starts as zeros (d_free phase 0); after each drain it is zeroed again
    // before the buffer is handed back, so every PV MMA accumulates.
    const uint32_t tdrow = tmem + C::kTmemD + ((uint32_t)(quarter * 32) << 16);
    auto zero_d = [&]() {
      tmem_zero80(tdrow);
      if constexpr (D == 128) tmem_zero64(tdrow + (C::kTmemDHi - C::kTmemD));
    };
    zero_d();
    tmem_wait_st();
    release_tmem(d_free, lane);
    for (int t = 0; t < nt; ++t) {
      if (!warp_wait(d_full, t & 1, wc)) break;
      tc_fence_after();
      const uint32_t taddr = tmem + C::kTmemD + ((uint32_t)(quarter * 32) << 16);
      const int qrow0 = (w.q_tile0 + t) * kSwBQ + quarter * 32;   // first query row of this warp's box
      const int grow0 = w.bh * Tp + qrow0;                        // its row in the [BH * Tp, d + 4] view of acc
      float a[32], rs;
      tmem_ld32(taddr, a);
      tmem_wait_ld_r(a);
      stage_box(a, 0, grow0);
      tmem_ld32(taddr + 32, a);
      tmem_ld1(taddr + 64, rs);
      tmem_wait_ld_r(a);
      tmem_wait_ld();
      if constexpr (D == 128) {
        stage_box(a, 32, grow0);
        const uint32_t thi = taddr + (C::kTmemDHi - C::kTmemD);
        tmem_ld32(thi, a);
        tmem_wait_ld_r(a);
        stage_box(a, 64, grow0);
        tmem_ld32(thi + 32, a);
        tmem_wait_ld_r(a);
      }
      zero_d();
      tmem_wait_st();
      release_tmem(d_free, lane);
      stage_box(a, D - 32, grow0);
      if (qrow0 + lane < T) atomicAdd(acc + ((size_t)grow0 + lane) * AS + D, rs);
    }
    if (lane == 0) bulk_wait_all();
  } else {
    // ----------------------------------------------------- demand warpgroups
    regs_inc_demand();
    const int g = wg;
    const int quarter = warp % 4;
    const int row = quarter * 32 + lane;            // key row inside the key tile
    const int kbase = w.key0 + g * kTile;           // first key of this warpgroup's tile
    const int swz = row % 8;
    const uint32_t tb = tmem + g * kTile + ((uint32_t)(quarter * 32) << 16);
    uint8_t *sh_row = sSh + g * kShBytes + (row / 8) * 1024 + (row % 8) * 128;
    float ceps = eps;   // committed + eps: demand this key received from earlier queries
    if (g == 0) {
      // this thread's key row (d bf16 = d / 2 words; zeros past T) -> TMEM
      // lane, 32 columns at a time
      const int64_t key = (int64_t)kbase + row;
      const uint4 *src = kglob + ((size_t)w.bh * T + key) * (D * 2 / 16);
#pragma unroll
      for (int part = 0; part < D / 64; ++part) {
        uint32_t kr[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const uint4 x = key < T ? __ldg(src + 8 * part + i) : make_uint4(0u, 0u, 0u, 0u);
          kr[4 * i] = x.x;
          kr[4 * i + 1] = x.y;
          kr[4 * i + 2] = x.z;
          kr[4 * i + 3] = x.w;
        }
        tmem_st32(tmem + C::kTmemK0 + 32 * part + ((uint32_t)(quarter * 32) << 16), kr);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(k0_full);
    }
    // 32 shares (bf16 pairs) of query chunk c -> 64-query M-block c/2, 16-byte
    // pieces (c%2)*4 .. +3 of this key's row, 128B-swizzled by row.
    auto store = [&](const uint32_t (&pk)[16], int c) {
      uint8_t *dst = sh_row + (c >> 1) * 16384;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        *reinterpret_cast<uint4 *>(dst + ((((c & 1) * 4 + i) ^ swz) * 16)) =
            make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
    };
    for (int t = 0; t < nt; ++t) {
      const int qlo = (w.q_tile0 + t) * kSwBQ;      // first query of the tile
      const bool all_masked = kbase > qlo + kSwBQ - 1 || kbase >= T;
      const bool need_mask = kbase + kTile - 1 > qlo;
      const int row_eff = row - (qlo - kbase);      // key after query col iff row_eff > col
      // Demand checkpoints for the backward (cchk != null): committed + eps of
      // this key at the start of each 32-query chunk, [bh][chunk][key < Tp]
      // (the last span can reach past Tp).
      float *ck = (!CHK || kbase + row >= Tp) ? nullptr : cchk + ((size_t)w.bh * (Tp / 32) + qlo / 32) * Tp + kbase + row;
      if (!warp_wait(&s_full[g], t & 1, wc)) break;
      tc_fence_after();
      uint32_t pk[16];
      if (all_masked) {
        if (CHK && ck != nullptr) {
#pragma unroll
          for (int c = 0; c < 4; ++c) ck[(size_t)c * Tp] = ceps;
        }
        release_tmem(&s_free[g], lane);
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = 0u;
        if (!warp_wait(&sh_free[g], (t & 1) ^ 1, wc)) break;
#pragma unroll
        for (int c = 0; c < 4; ++c) store(pk, c);
      } else {
        // 32-column chunks; the load of chunk c+1 is in flight while chunk c is formed.
        float A[32], B[32];
        tmem_ld32(tb, A);
        tmem_wait_ld_r(A);
        tmem_ld32(tb + 32, B);
        if (CHK && ck != nullptr) ck[0 * (size_t)Tp] = ceps;
        if (need_mask) demand_chunk<true, 0, EARLIER>(A, row_eff, c2, ceps, pk);
        else demand_chunk<false, 0, EARLIER>(A, row_eff, c2, ceps, pk);
        // the product of the previous query tile must be done reading this buffer
        if (!warp_wait(&sh_free[g], (t & 1) ^ 1, wc)) break;
        store(pk, 0);
        tmem_wait_ld_r(B);
        tmem_ld32(tb + 64, A);
        if (CHK && ck != nullptr) ck[1 * (size_t)Tp] = ceps;
        if (need_mask) demand_chunk<true, 1, EARLIER>(B, row_eff, c2, ceps, pk);
        else demand_chunk<false, 1, EARLIER>(B, row_eff, c2, ceps, pk);
        store(pk, 1);
        tmem_ld32(tb + 96, B);
        tmem_wait_ld_r(A);
        tmem_wait_ld_r(B);
        release_tmem(&s_free[g], lane);   // the next tile's S runs while the last two chunks are formed
        if (CHK && ck != nullptr) ck[2 * (size_t)Tp] = ceps;
        if (need_mask) demand_chunk<true, 2, EARLIER>(A, row_eff, c2, ceps, pk);
        else demand_chunk<false, 2, EARLIER>(A, row_eff, c2, ceps, pk);
        store(pk, 2);
        if (CHK && ck != nullptr) ck[3 * (size_t)Tp] = ceps;
        if (need_mask) demand_chunk<true, 3, EARLIER>(B, row_eff, c2, ceps, pk);
        else demand_chunk<false, 3, EARLIER>(B, row_eff, c2, ceps, pk);
        store(pk, 3);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sh_full[g]);
      }
    }
    const int64_t key = (int64_t)kbase + row;
    if (demand_out != nullptr && key < T && !*abort_flag) demand_out[(size_t)w.bh * T + key] = ceps - eps;
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ============================================================================
// Host side
// ============================================================================
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (fn == nullptr) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// [BH, T, d] bf16 viewed as a 3-D tensor; box = 64 columns (one half) of
// one tile of `rows` rows of one head.  Rows past T read as zero.
static bool make_tile_map(CUtensorMap *m, const void *base, int BH, int T, int d, int rows = kTile) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)T, (cuuint64_t)BH};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)T * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// For the backward's kernels.
bool make_bf16_tile_map(CUtensorMap *m, const void *base, int BH, int T, int d, int rows) {
  return make_tile_map(m, base, BH, T, d, rows);
}

// The fp32 accumulator [BH * Tp rows][d + 4] as a 2-D tensor; box = 32 rows
// x 32 columns, 128B swizzle: the sweep epilogue's reduction box.
static bool make_acc_map(CUtensorMap *m, float *acc, int64_t rows, int d) {
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)acc_stride(d), (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)acc_stride(d) * 4};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, acc, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_finalize_bf16(const float *acc, const float *lse2_ws, __nv_bfloat16 *out, float *rowsum_out,
                                 float *lse2_out, int BH, int T, int d, cudaStream_t stream);

// Shared-memory opt-in and register-split check of one sweep instantiation.
template <int D, bool EARLIER, bool CHK>
static int prepare_sweep() {
  using C = SwCfg<D>;
  if (cudaFuncSetAttribute(sweep_kernel<D, EARLIER, CHK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           C::kSmemBytes) != cudaSuccess)
    return DA_ERR_CUDA;
  // The sweep's warpgroups re-split the block's registers (setmaxnreg); a
  // split larger than what the block is launched with would never resolve,
  // so refuse to launch unless the compiled register count covers it.
  cudaFuncAttributes fa;
  if (cudaFuncGetAttributes(&fa, sweep_kernel<D, EARLIER, CHK>) != cudaSuccess) return DA_ERR_CUDA;
  if (fa.numRegs * C::kThreads < C::kRegsNeeded || fa.numRegs > kSwRegsDemand || fa.numRegs < kSwRegsEpi)
    return DA_ERR_UNSUPPORTED;
  return DA_OK;
}

template <int D>
static int prepare_fwd_bf16() {
  if (cudaFuncSetAttribute(rowstats_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           RsCfg<D>::kSmemBytes) != cudaSuccess)
    return DA_ERR_CUDA;
  int st = prepare_sweep<D, false, false>();
  if (st == DA_OK) st = prepare_sweep<D, true, false>();
  if (st == DA_OK) st = prepare_sweep<D, false, true>();   // the backward's forward-again sweep
  if (st == DA_OK) st = prepare_sweep<D, true, true>();
  return st;
}

// The per-device set-up of the forward kernels of head dimension D, shared
// by the forward and the backward's forward-again sweep.
template <int D>
static PerDeviceOnce &fwd_bf16_once() {
  static PerDeviceOnce once;
  return once;
}

// Blocks of the fix-up pass (two per SM of a GB300; grid-stride over rows).
constexpr int kFixupBlocks = 304;
template <int D>
static int launch_fwd_bf16_t(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                             const CUtensorMap &ta, const void *q, const void *k, float *demand_out, int BH, int T,
                             HeadScale hs,
                             float eps, bool earlier, float *lse2_ws, float *acc, float *cchk, int *status,
                             cudaStream_t stream, cudaEvent_t const *ev) {
  // The shared-memory opt-in is a per-device function attribute.
  const int prep = fwd_bf16_once<D>().run(prepare_fwd_bf16<D>);
  if (prep != DA_OK) return prep;
  using C = SwCfg<D>;
  const int Tp = (int)t_pad(T);
  if (ev[0]) cudaEventRecord(ev[0], stream);
  rowstats_kernel<D><<<rowstats_num_ctas(BH, T), kRsThreads, RsCfg<D>::kSmemBytes, stream>>>(tq, tk, lse2_ws, acc,
                                                                                            BH, T, Tp, hs, status);
  rowstats_fixup_kernel<D><<<kFixupBlocks, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(q),
                                                              static_cast<const __nv_bfloat16 *>(k), lse2_ws, BH, T,
                                                              Tp, hs, status);
  if (ev[1]) cudaEventRecord(ev[1], stream);
  const int nsw = sweep_num_ctas(BH, T, D);
  const uint4 *kg = static_cast<const uint4 *>(k);
  // cchk != null: also keep the demand checkpoints for a later backward
#define DA_SWEEP_ARGS tq, tk, tv, ta, kg, lse2_ws, acc, demand_out, cchk, BH, T, Tp, hs, eps, status
  if (cchk != nullptr) {
    if (earlier) sweep_kernel<D, true, true><<<nsw, C::kThreads, C::kSmemBytes, stream>>>(DA_SWEEP_ARGS);
    else sweep_kernel<D, false, true><<<nsw, C::kThreads, C::kSmemBytes, stream>>>(DA_SWEEP_ARGS);
  } else {
    if (earlier) sweep_kernel<D, true, false><<<nsw, C::kThreads, C::kSmemBytes, stream>>>(DA_SWEEP_ARGS);
    else sweep_kernel<D, false, false><<<nsw, C::kThreads, C::kSmemBytes, stream>>>(DA_SWEEP_ARGS);
  }
#undef DA_SWEEP_ARGS
  if (cudaGetLastError() != cudaSuccess) return DA_ERR_CUDA;
  return DA_OK;
}

// The demand sweep alone, for the backward: the caller has written -lse2 to
// nlse2 and zeroed acc; cchk receives the demand checkpoints.
template <int D>
static int launch_sweep_chk_t(const void *q, const void *k, const void *v, const float *nlse2, float *acc,
                              float *cchk, int BH, int T, HeadScale hs, float eps, bool earlier, int *status,
                              cudaStream_t stream) {
  const int64_t acc_rows = (int64_t)BH * (int64_t)t_pad(T);
  if (acc_rows > 0x7FFFFFFF) return DA_ERR_UNSUPPORTED;
  CUtensorMap tq, tk, tv, ta;
  if (!make_tile_map(&tq, q, BH, T, D) || !make_tile_map(&tk, k, BH, T, D) || !make_tile_map(&tv, v, BH, T, D) ||
      !make_acc_map(&ta, acc, acc_rows, D))
    return DA_ERR_CUDA;
  const int prep = fwd_bf16_once<D>().run(prepare_fwd_bf16<D>);
  if (prep != DA_OK) return prep;
  using C = SwCfg<D>;
  const int Tp = (int)t_pad(T);
  const int nsw = sweep_num_ctas(BH, T, D);
  const uint4 *kg = static_cast<const uint4 *>(k);
  if (earlier)
    sweep_kernel<D, true, true><<<nsw, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, ta, kg, nlse2, acc, nullptr,
                                                                             cchk, BH, T, Tp, hs, eps, status);
  else
    sweep_kernel<D, false, true><<<nsw, C::kThreads, C::kSmemBytes, stream>>>(tq, tk, tv, ta, kg, nlse2, acc,
                                                                              nullptr, cchk, BH, T, Tp, hs, eps,
                                                                              status);
  return cudaGetLastError() == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

int launch_sweep_bf16_chk(const void *q, const void *k, const void *v, const float *nlse2, float *acc, float *cchk,
                          int BH, int T, int d, HeadScale hs, float eps, bool earlier, int *status,
                          cudaStream_t stream) {
  return d == 128 ? launch_sweep_chk_t<128>(q, k, v, nlse2, acc, cchk, BH, T, hs, eps, earlier, status, stream)
                  : launch_sweep_chk_t<64>(q, k, v, nlse2, acc, cchk, BH, T, hs, eps, earlier, status, stream);
}

int launch_fwd_bf16(const void *q, const void *k, const void *v, void *out, float *lse2_out, float *rowsum_out,
                    float *demand_out, int BH, int T, int d, HeadScale hs, float eps, bool earlier, float *lse2_ws,
                    float *acc, float *cchk, int *status, cudaStream_t stream, cudaEvent_t const *ev) {
  const int64_t acc_rows = (int64_t)BH * (int64_t)t_pad(T);
  if (acc_rows > 0x7FFFFFFF) return DA_ERR_UNSUPPORTED;   // TMA row coordinates are 32-bit
  CUtensorMap tq, tk, tv, ta;
  if (!make_tile_map(&tq, q, BH, T, d) || !make_tile_map(&tk, k, BH, T, d) || !make_tile_map(&tv, v, BH, T, d) ||
      !make_acc_map(&ta, acc, acc_rows, d))
    return DA_ERR_CUDA;
  const int st = d == 128 ? launch_fwd_bf16_t<128>(tq, tk, tv, ta, q, k, demand_out, BH, T, hs, eps, earlier, lse2_ws,
                                                   acc, cchk, status, stream, ev)
                          : launch_fwd_bf16_t<64>(tq, tk, tv, ta, q, k, demand_out, BH, T, hs, eps, earlier, lse2_ws,
                                                  acc, cchk, status, stream, ev);
  if (st != DA_OK) return st;
  if (ev[2]) cudaEventRecord(ev[2], stream);
  if (launch_finalize_bf16(acc, lse2_ws, reinterpret_cast<__nv_bfloat16 *>(out), rowsum_out, lse2_out, BH, T, d,
                           stream) != cudaSuccess)
    return DA_ERR_CUDA;
  if (ev[3]) cudaEventRecord(ev[3], stream);
  return DA_OK;
}

}  // namespace da
