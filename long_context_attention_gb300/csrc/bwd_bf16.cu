// Tensor-core backward of dilution attention (bf16, d = 64 and d = 128).
//
// Gradients of sum(dout * out) through the operator of "DilutionAttention
// v0.1.0 · results", section "The operator" (the page states only that exact
// gradients exist; the chain rule is written out in bwd.cu).  Per (batch,
// head), with g = dout, r = share, R_j = sum_k r_jk, D = committed + p + eps
// (committed + eps for the earlier-demand-only variant):
//   dA'_jk = g_j . v_k - delta_j,          delta_j = g_j . out_j
//   dr_jk  = dA'_jk / R_j
//   dC_jk  = -dr_jk p_jk / D_jk^2          dp_jk = direct_jk + sum_{i > j} dC_ik
//   direct = dr (committed + eps) / D^2    (dr / D for the variant)
//   rho_j  = sum_k p_jk dp_jk,             ds_jk = p_jk (dp_jk - rho_j)
//   dV_k   = sum_j (r_jk / R_j) g_j,  dK_k = c sum_j ds_jk q_j,  dQ_j = c sum_k ds_jk k_k
//
// Every pair (j, k) needs the forward running sum down its key column
// (committed) and the reverse running sum of dC, and rho needs a reduction
// over all keys before any ds exists.  Since ds = p (dp - rho),
//   dK_k = c (sum_j u_jk q_j - sum_j p_jk rho_j q_j),  u = p dp,
// and only the second sum needs rho.  The passes:
//   F   the forward demand sweep again (fwd_bf16.cu) from the given lse2; it
//       writes committed + eps of every key at every 32-query chunk start
//       (demand checkpoints) and the forward accumulators (numerator, R);
//   rows  from those accumulators, per query row: Gs = G / R (the upstream
//       gradient over the row sum of the shares, bf16) and delta / R with
//       delta_j = g_j . out_j;
//   R   key-major, query chunks in reverse order: S = K Q^T and
//       dr = V Gs^T - delta / R on tcgen05; one thread per key rebuilds
//       committed inside each chunk from its checkpoint, carries
//       sum_{i > j} dC in a register, and writes it at every chunk start
//       (reverse checkpoints); it forms the shares r and u = p dp, tcgen05
//       accumulates dV += r^T Gs (= A^T G, A = r / R) and dK1 += u^T Q in
//       TMEM, and rho_j (the sum of u over the key tile's lanes) is added to
//       rho;
//   L   key-major, no demand: the bids p again (S product, one exponential
//       per pair), dK2 += (p rho)^T Q on tcgen05, dK = c (dK1 - dK2);
//   Q   query-major: with both checkpoints every chunk is independent; for
//       each key tile the threads write ds (MN-major) and tcgen05 accumulates
//       dQ += ds K in TMEM.
// S and dA' are formed 64 queries at a time (N = 64) so two CTAs fit an SM
// at d = 64 (R at d = 128: one, its tiles and N = 128 accumulators take the
// SM); -lse2 / c2 and -delta / R ride in a fifth K step of their products
// (the extension operands of the forward sweep).  The passes' launch orders are
// bwd_work's (da_internal.h): heads in groups whose streamed tiles stay in
// L2.  Every wait is bounded.
#include "da_internal.h"
#include "da_ptx.cuh"

#include <cuda.h>
#include <cuda_bf16.h>



namespace da {

namespace {

constexpr int kBtThreads = 192;                    // 4 demand warps, producer, MMA issuer

// R at d = 64 re-splits its registers (setmaxnreg): warpgroup 0 (the key
// warps) takes 224 per thread, warpgroup 1 (producer, issuer and two idle
// warps that complete it) gives up to 32; launched at 128 per thread (two CTAs
// of 256 threads per SM), the split uses exactly the block's registers
// (216 / 40 measured 0.03 ms slower, 232 / 24 spills in warpgroup 1).  (At
// 168 for every warp the key warps spilled; backward 13.754 -> 13.711 ms, and
// the room lets the two-chunk loop unroll.)  The same split in the dQ pass
// measured 0.15 ms slower.
template <int D>
struct RevRegs {
  static constexpr bool kSplit = D == 64;
  static constexpr int kThreads = kSplit ? 256 : kBtThreads;
  static constexpr int kLaunch = kSplit ? 128 : 0;
  static constexpr int kKey = 224, kCtl = 32;
  static constexpr int kNeeded = 128 * (kKey + kCtl);
  static_assert(!kSplit || kNeeded <= kThreads * kLaunch, "register split exceeds the launch registers");
};
template <int N>
__device__ __forceinline__ void setmaxnreg_inc() { asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N)); }
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() { asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N)); }
// A tile of R rows x d bf16 is stored as d / 64 column halves of R rows x 64
// (128-byte swizzled rows), R * 128 bytes each.
constexpr uint32_t kH128 = kTile * 64 * 2;         // one half of a 128-row tile
constexpr uint32_t kH64 = 64 * 64 * 2;             // one half of a 64-row tile
constexpr uint32_t kExt128 = 128 * 16 * 2;         // extension operand, 128 rows
constexpr uint32_t kExt64 = 64 * 16 * 2;           // extension operand, 64 rows

constexpr uint32_t round_up_c(uint32_t x, uint32_t m) { return (x + m - 1) / m * m; }

__device__ __forceinline__ uint64_t kdesc(const uint8_t *tile, int kstep) {
  return smem_desc(smem_u32(tile) + kstep * 32, 16, 1024);
}

// TMA load of one R-row tile of a [BH, T, d] tensor, half by half (the maps
// have 64-column boxes of R rows).
template <int D, uint32_t HALF>
__device__ __forceinline__ void load_tile_halves(uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int row, int bh) {
#pragma unroll
  for (int h = 0; h < D / 64; ++h) tma_load_3d(dst + h * HALF, map, bar, h * 64, row, bh);
}

__device__ __forceinline__ void drain_wait_bt(uint64_t *bar, uint32_t parity) {
  const unsigned long long t0 = globaltimer();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer() - t0 > 100ull * 1000ull * 1000ull) break;
  }
}

__device__ __forceinline__ void release_bt(uint64_t *bar, int lane) {
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
}

// Extension operand rows (K-major, no swizzle: 8-row groups of 256 bytes,
// each the core matrix of K 0..7 then that of K 8..15): row q = [hi mid lo 0
// ...] of v, the bf16 parts of an fp32 value (24 significant bits).  Rows of
// queries past T carry a large finite negative value (their bids vanish).
__device__ __forceinline__ void put_ext_row(uint8_t *ext, int q, float v) {
  v = fmaxf(v, -3.0e38f);
  const __nv_bfloat16 h = __float2bfloat16_rn(v);
  const float r1 = v - __bfloat162float(h);
  const __nv_bfloat16 m = __float2bfloat16_rn(r1);
  const __nv_bfloat16 l = __float2bfloat16_rn(r1 - __bfloat162float(m));
  *reinterpret_cast<uint4 *>(ext + (q >> 3) * 256 + (q & 7) * 16) =
      make_uint4((uint32_t)__bfloat16_as_ushort(h) | ((uint32_t)__bfloat16_as_ushort(m) << 16),
                 (uint32_t)__bfloat16_as_ushort(l), 0u, 0u);
}

// Zero `bytes` of shared memory (the extension rows' K 8..15 core matrices
// are never rewritten: they must hold zeros, not stale bits, since 0 x Inf
// would reach the products).
__device__ __forceinline__ void zero_smem(uint8_t *p, uint32_t bytes, int tid, int nthreads) {
  for (uint32_t e = tid; e < bytes / 16; e += nthreads) reinterpret_cast<uint4 *>(p)[e] = make_uint4(0u, 0u, 0u, 0u);
}

// A_ext: [1 1 1 0 ...] for every one of 128 rows; its zero half K 8..15 too.
__device__ __forceinline__ void fill_ones_ext(uint8_t *ext, int tid, int nthreads) {
  for (int e = tid; e < (int)(kExt128 / 16); e += nthreads) {
    const bool k_lo = (e & 15) < 8;
    reinterpret_cast<uint4 *>(ext)[e] = k_lo ? make_uint4(0x3F803F80u, 0x00003F80u, 0u, 0u) : make_uint4(0u, 0u, 0u, 0u);
  }
}

}  // namespace

// ---------------------------------------------------------------- prep / rows
// -lse2 for the sweep (rows past T: -inf) and zeroed forward accumulators.
template <int D>
__global__ void bwdtc_prep(const float *__restrict__ lse2, float *__restrict__ nlse2, float *__restrict__ acc,
                           int BH, int T, int Tp) {
  const int64_t row = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (row >= (int64_t)BH * Tp) return;
  const int64_t bh = row / Tp, i = row % Tp;
  nlse2[row] = i < T ? -lse2[bh * T + i] : -INFINITY;
  float4 *ar = reinterpret_cast<float4 *>(acc + row * acc_stride(D));
#pragma unroll
  for (int t = 0; t < acc_stride(D) / 4; ++t) ar[t] = make_float4(0.f, 0.f, 0.f, 0.f);
}

// Per query row j: gs_j = g_j / R_j (bf16), delta_j / R_j with delta_j =
// g_j . out_j (out = numerator / R), and rho_j = 0; 16 threads per row, d / 16
// columns each.  Rows past T get zeros, so their dr vanish.
template <int D>
__global__ void bwdtc_rows(const float *__restrict__ acc, const __nv_bfloat16 *__restrict__ g,
                           __nv_bfloat16 *__restrict__ gs, float *__restrict__ delta, float *__restrict__ rho,
                           int BH, int T, int Tp) {
  const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = t / 16;
  const int part = (int)(t % 16);
  const bool live = row < (int64_t)BH * Tp;
  const int64_t bh = live ? row / Tp : 0, i = live ? row % Tp : 0;
  float dot = 0.f, inv = 0.f;
  if (live && i < T) {
    const float *ar = acc + row * acc_stride(D);
    inv = 1.f / ar[D];
#pragma unroll
    for (int j = 0; j < D / 64; ++j) {
      const float4 a = reinterpret_cast<const float4 *>(ar)[part + 16 * j];
      const uint2 gg = reinterpret_cast<const uint2 *>(g + (bh * T + i) * D)[part + 16 * j];
      const float2 g01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gg.x));
      const float2 g23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&gg.y));
      dot += (a.x * g01.x + a.y * g01.y) + (a.z * g23.x + a.w * g23.y);
      reinterpret_cast<uint2 *>(gs + (bh * T + i) * D)[part + 16 * j] =
          make_uint2(pack_bf16x2(g01.x * inv, g01.y * inv), pack_bf16x2(g23.x * inv, g23.y * inv));
    }
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
  if (live && part == 0) {
    delta[row] = dot * inv * inv;
    rho[row] = 0.f;
  }
}

// ------------------------------------------------------------- chunk engine
// One key (this thread) against 32 consecutive queries q0 .. q0 + 31 of its
// column.  In: S' (q.k - lse2 / c2) and dr = (g.v - delta) / R from TMEM (the
// product takes g / R and delta / R), and the chunk's demand checkpoint
// cpe = committed + eps before q0.  Forms, for each query in causal order, p,
// D = e + p with e = committed + eps before the query (D is the running sum
// just after the query; for EARLIER D = e, just before it), the share
// r = p / D and
//   dr / D,   -dC = (dr / D) r,
// leaving p in P, dr / D in A and -dC in E (and, with AT, r packed as bf16
// pairs).  The direct term of dp, dr e / D^2 = dr / D + dC, needs no product
// of its own: the reverse walk adds the running sum of dC including the
// query's own (for EARLIER the direct term is dr / D itself).  (Taking D from
// the running sum instead of adding e + p again: backward 11.09 -> 10.98 ms.)
// (Forming dr e / D^2 per pair: backward 11.40 ms at 4x12x16384x64 against
// 11.09 ms without; folding -rho into it by a fused multiply-add in the dQ
// pass spilled there.)  Pairs of queries share one reciprocal, 1 / (D0 D1), and go
// through the packed f32x2 pipe.  MASK zeroes keys after the query
// (row_eff > column).  (With dout and delta in the products and 1/R read per
// query pair from shared memory the backward took 12.32 ms at 4x12x16384x64,
// with dout / R 11.65 ms; a reciprocal per query instead of one per pair
// 11.75 ms.)
template <bool MASK, bool EARLIER, bool AT>
__device__ __forceinline__ void bwd_chunk_fwd(float (&P)[32], float (&A)[32], float (&E)[32], uint32_t (&at)[16],
                                              int row_eff, int col0, float c2, float cpe) {
  const float2 c2v = make_float2(c2, c2);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 x = fmul2(make_float2(P[i], P[i + 1]), c2v);
    P[i] = ex2_approx(x.x);
    P[i + 1] = ex2_approx(x.y);
  }
  if (MASK) {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (row_eff > col0 + i) P[i] = 0.f;
  }
  // D of each query straight from the running sum: committed + eps after the
  // query (committed + eps + p), or before it for EARLIER
  // (stored pairwise swapped, E[2 i] holding D of query 2 i + 1, so that the
  // pair (1/D0, 1/D1) = (D1, D0) / (D0 D1) is one packed product)
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (EARLIER) {
      E[i ^ 1] = cpe;
      cpe += P[i];
    } else {
      cpe += P[i];
      E[i ^ 1] = cpe;
    }
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 p = make_float2(P[2 * i], P[2 * i + 1]);
    const float2 ds = make_float2(E[2 * i], E[2 * i + 1]);   // (D1, D0)
    const float rr = rcp_approx(ds.x * ds.y);
    const float2 inv = fmul2(ds, make_float2(rr, rr));          // 1/D0, 1/D1
    float2 dri = fmul2(make_float2(A[2 * i], A[2 * i + 1]), inv);            // dr / D
    if (MASK) {
      if (row_eff > col0 + 2 * i) dri.x = 0.f;
      if (row_eff > col0 + 2 * i + 1) dri.y = 0.f;
    }
    const float2 r = fmul2(p, inv);     // the share p / D
    const float2 ndc = fmul2(dri, r);   // -dC = dr p / D^2
    if (AT) at[i] = pack_bf16x2(r.x, r.y);
    A[2 * i] = dri.x;
    A[2 * i + 1] = dri.y;
    E[2 * i] = ndc.x;
    E[2 * i + 1] = ndc.y;
  }
}

// Reverse walk of one chunk (queries in reverse order; E holds -dC, A dr / D):
// grev += dC, then dp = dr / D + grev (the sum of dC over this query and the
// later ones); for EARLIER dp = dr / D + grev before this query's dC.  dp is
// left in A.  The running sum is the only serial chain; the additions into A
// go two at a time on the packed pipe (backward 12.36 -> 12.30 ms with the
// dQ pass's rho kept negated).
template <bool EARLIER>
__device__ __forceinline__ void bwd_chunk_rev(float (&A)[32], const float (&E)[32], float &grev) {
  float G[32];
#pragma unroll
  for (int i = 31; i >= 0; --i) {
    if (EARLIER) {
      G[i] = grev;
      grev -= E[i];
    } else {
      grev -= E[i];
      G[i] = grev;
    }
  }
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 a = fadd2(make_float2(A[i], A[i + 1]), make_float2(G[i], G[i + 1]));
    A[i] = a.x;
    A[i + 1] = a.y;
  }
}

// ------------------------------------------------------------ key-major passes
// One CTA per (head, 128-key tile), two per SM at d = 64.  Warps 0-3: one
// thread per key; warp 4: TMA and the per-query extension rows; warp 5: MMA
// issuer.
//
// R (bwdtc_rev_kernel) walks the key tile's 64-query half tiles from the last
// one back to the diagonal.  Per half tile: S' = K Q^T and dA' = V G^T - delta
// on tcgen05; one thread per key rebuilds committed inside each 32-query
// chunk from its demand checkpoint, carries the reverse sum of dC (writing it
// at every chunk start: the reverse checkpoints), and forms
//   r = p / D (bf16, for dV),   u = p dp (bf16, for dK1; for rho: bf16 at
//   d = 64, where the warp sums read the u^T operand back, fp32 at d = 128);
// the products dV += r^T Gs and dK1 += u^T Q accumulate in TMEM, and the
// key tile's partial sums of u (rho_j = sum_k p_jk dp_jk) go to rho.
// Because ds = p (dp - rho),
//   dK_k = c sum_j ds_jk q_j = c (sum_j u_jk q_j - sum_j p_jk rho_j q_j),
// so the rest of dK needs rho but not the demand: L (bwdtc_dk2_kernel) forms
// the bids p again (S' product, one exponential per pair) and accumulates
// dK2 += (p rho)^T Q, then writes dK = c (dK1 - dK2).
constexpr int kModeRev = 0, kModeDk2 = 1;

template <int MODE, int D>
struct KeyCfg {
  static constexpr uint32_t kTB = kTile * D * 2, kHB = 64 * D * 2;   // 128-row and 64-row tiles
  static constexpr bool kRev = MODE == kModeRev;
  static constexpr uint32_t kOffK = 0;
  static constexpr uint32_t kOffV = kOffK + kTB;                          // R only
  static constexpr uint32_t kOffQh = kRev ? kOffV + kTB : kOffK + kTB;    // [2] 64-query tiles of Q
  static constexpr uint32_t kOffGh = kOffQh + 2 * kHB;                    // [2] 64-query tiles of dout (R)
  static constexpr uint32_t kOffAExt = kRev ? kOffGh + 2 * kHB : kOffGh;
  static constexpr uint32_t kOffBExtS = kOffAExt + kExt128;               // [2] -lse2 / c2 rows
  static constexpr uint32_t kOffBExtA = kOffBExtS + 2 * kExt64;           // [2] -delta rows (R)
  static constexpr uint32_t kOffRows = kOffBExtA + (kRev ? 2 * kExt64 : 0);   // [2][64] fp32: rho (L)
  static constexpr uint32_t kOffRed = kOffRows + 2 * 64 * 4;              // [2][4][64] fp32 partial rho (R)
  static constexpr uint32_t kOffOp = round_up_c(kOffRed + (kRev ? 2 * 4 * 64 * 4 : 0), 1024);
  // R: A^T and u^T (bf16, K-major: 128 keys x 64 queries, 128B-swizzled);
  // L: two buffers of (p rho)^T
  // R at d = 128 (one CTA per SM) has room for the per-warp transposition
  // buffers of the partial rho sums, [4][32][36] fp32; at d = 64 they would
  // not fit beside the second CTA and a register butterfly does the sums.
  static constexpr bool kXp = kRev && D == 128;
  static constexpr uint32_t kOffXp = kOffOp + 2 * kH128;
  static constexpr uint32_t kOffBar = kOffXp + (kXp ? 4 * 32 * 36 * 4 : 0);
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;         // + re-alignment slack
  // TMEM: S' (and dA'), then the accumulators (d columns each):
  //   R: S' 0..63, dA' 64..127, dV, dK1;   L: S' 0..63, dK2
  // (L at d = 64 runs three CTAs per SM: 128 columns each)
  static constexpr uint32_t kTmemAcc0 = kRev ? 128 : 64, kTmemAcc1 = kTmemAcc0 + D;
  static constexpr uint32_t kTmemCols = kRev ? (D == 128 ? 512 : 256) : (D == 128 ? 256 : 128);
  static constexpr int kCtasPerSm = kRev ? (D == 128 ? 1 : 2) : (D == 128 ? 2 : 3);
  static_assert(kOffOp % 1024 == 0, "swizzled operands");
  static_assert(kSmemBytes * kCtasPerSm <= 232448, "shared memory");
};

// The K-major S' = K Q^T (or dA' = V G^T) product over d: K steps 0..3 read
// the first 64 columns of both operands, 4..7 (d = 128) the second halves.
template <int D>
__device__ __forceinline__ void mma_over_d(uint32_t dt, uint64_t da, uint32_t half_a, uint64_t db, uint32_t half_b,
                                           uint32_t idesc) {
  MmaRun<0, 4, 2, 2, false>::go(dt, da, db, idesc, 0u);
  if constexpr (D == 128) MmaRun<0, 4, 2, 2, false>::go(dt, da + (half_a >> 4), db + (half_b >> 4), idesc, 1u);
}

// The sums over the warp's 32 keys of u for the half tile's 64 queries, read
// back from the warp's 32 rows of the u^T operand (bf16, 128-byte rows whose
// 16-byte pieces are swizzled by the row index mod 8): lane l adds up queries
// 2 l and 2 l + 1, one 4-byte word per row (the 32 lanes read a whole row,
// free of bank conflicts).  The bf16 values are the ones the dK1 product
// takes, so sum_k u_jk - rho_j sum_k p_jk stays zero up to the fp32 sums.
// Each bf16 half is added into its fp32 sum by a mixed-precision add (the
// conversion is exact): backward 10.97 -> 10.92 ms at 4x12x16384x64 against
// unpacking both halves and one packed add, together with the pairwise
// swapped D in the chunk engine.  (The fp32 sums by a register butterfly --
// five rounds of shuffles, each lane keeping one half -- took about 110
// instructions per 32-query chunk against about 65 with the unpacking:
// backward 12.45 -> 12.36 ms.  The rounding of u to bf16 moves rho by about
// 2^-9 of its terms' spread, under 0.3 % of max |dQ| in the float64 model
// of it.)
__device__ __forceinline__ void add_bf16x2(float &lo_acc, float &hi_acc, uint32_t x) {
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(lo_acc), "+f"(hi_acc)
      : "r"(x));
}
__device__ __forceinline__ float2 ut_column_sums(const uint8_t *rows, int lane) {
  float s0[4] = {}, s1[4] = {};
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const uint32_t x = *reinterpret_cast<const uint32_t *>(
        rows + (i >> 3) * 1024 + (i & 7) * 128 + ((((lane >> 2) ^ (i & 7)) << 4) | ((lane & 3) << 2)));
    add_bf16x2(s0[i & 3], s1[i & 3], x);
  }
  return make_float2((s0[0] + s0[1]) + (s0[2] + s0[3]), (s1[0] + s1[1]) + (s1[2] + s1[3]));
}

// The same sums through shared memory: each lane writes its 32 values as one
// row of the warp's [32][36] block (the row pitch of 36 words keeps both the
// 16-byte row stores and the column reads free of bank conflicts), then lane l
// adds up column l.
__device__ __forceinline__ float warp_column_sum(const float (&X)[32], float *red, int lane) {
  float *rowp = red + lane * 36;
#pragma unroll
  for (int j = 0; j < 8; ++j)
    *reinterpret_cast<float4 *>(rowp + 4 * j) = make_float4(X[4 * j], X[4 * j + 1], X[4 * j + 2], X[4 * j + 3]);
  __syncwarp();
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
  for (int r = 0; r < 32; r += 4) {
    s0 += red[r * 36 + lane];
    s1 += red[(r + 1) * 36 + lane];
    s2 += red[(r + 2) * 36 + lane];
    s3 += red[(r + 3) * 36 + lane];
  }
  __syncwarp();   // the block is free again
  return (s0 + s1) + (s2 + s3);
}

template <int D, bool EARLIER>
__global__ void __launch_bounds__(RevRegs<D>::kThreads, KeyCfg<kModeRev, D>::kCtasPerSm)
    bwdtc_rev_kernel(const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmGh,
                     const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                     const float *__restrict__ nlse2, const float *__restrict__ delta,
                     float *__restrict__ rho, const float *__restrict__ cchk,
                     float *__restrict__ gchk, float *__restrict__ dk1, __nv_bfloat16 *__restrict__ dv, int BH,
                     int T, int Tp, HeadScale hs, int *status) {
  using C = KeyCfg<kModeRev, D>;
  extern __shared__ uint8_t bt_smem_raw[];
  uint8_t *smem = bt_smem_raw + ((1024u - (smem_u32(bt_smem_raw) & 1023u)) & 1023u);
  uint8_t *sK = smem + C::kOffK, *sV = smem + C::kOffV;
  uint8_t *sAExt = smem + C::kOffAExt;
  float *sRed = reinterpret_cast<float *>(smem + C::kOffRed);
  uint8_t *sAT = smem + C::kOffOp, *sUT = smem + C::kOffOp + kH128;
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *kv_full = bars;
  uint64_t *in_full = bars + 1;      // [2] half tile b loaded and its rows written
  uint64_t *in_empty = bars + 3;     // [2] its products done and its rows read
  uint64_t *s_full = bars + 5;       // S' / dA' slot
  uint64_t *s_free = bars + 6;
  uint64_t *x_full = bars + 7;       // A^T, u^T of the half tile written
  uint64_t *x_free = bars + 8;       // dV, dK1 products of the half tile done
  uint64_t *r_full = bars + 9;       // [2] partial rho written
  uint64_t *r_free = bars + 11;      // [2] partial rho read
  uint64_t *fin = bars + 13;
  uint64_t *drain = bars + 14;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 15);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const TileWork tw = bwd_work(blockIdx.x, BH, T, D, kBwdRev);
  const int bh = tw.bh, kt = tw.q_tile0;
  const int NH = Tp / 64, hq0 = 2 * kt, n = NH - hq0, NC = Tp / 32;
  // as in the forward sweep: a scale of at least 1e-30 keeps -inf logits at -inf
  const float c2 = fmaxf(head_c2(hs, bh, nullptr), 1e-30f);

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&in_full[b], 2);    // the tiles' bytes + the producer's rows
      mbar_init(&in_empty[b], 5);   // the issuer's commit + the four key warps
      mbar_init(&r_full[b], 4);
      mbar_init(&r_free[b], 2);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(x_full, 4);
    mbar_init(x_free, 1);
    mbar_init(fin, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  fill_ones_ext(sAExt, threadIdx.x, RevRegs<D>::kThreads);
  zero_smem(smem + C::kOffBExtS, 4 * kExt64, threadIdx.x, RevRegs<D>::kThreads);   // both buffers of both rows
  fence_proxy_async_smem();
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, status};
  auto half_of = [&](int u) { return NH - 1 - u; };

  if (warp >= 4) {
    // warpgroup 1 (producer, issuer, and at d = 64 two idle warps that
    // complete it): one register re-split for all four warps
    if constexpr (RevRegs<D>::kSplit) setmaxnreg_dec<RevRegs<D>::kCtl>();
    if (warp == 4) {
      // -------------------------------------------------------- producer
      if (lane == 0) {
        prefetch_tmap(&tmQh);
        prefetch_tmap(&tmGh);
        prefetch_tmap(&tmK);
        prefetch_tmap(&tmV);
        mbar_arrive_expect_tx(kv_full, 2 * C::kTB);
        load_tile_halves<D, kH128>(sK, &tmK, kv_full, kt * kTile, bh);
        load_tile_halves<D, kH128>(sV, &tmV, kv_full, kt * kTile, bh);
      }
      int issued = 0;
      for (int u = 0; u < n; ++u) {
        const int b = u & 1, h = half_of(u);
        // the half tile's per-query values are read before waiting for the
        // buffer, so their global-memory latency overlaps that wait
        float nl[2], de[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const size_t idx = (size_t)bh * Tp + h * 64 + lane + 32 * j;
          nl[j] = __ldg(nlse2 + idx);
          de[j] = __ldg(delta + idx);
        }
        if (!mbar_wait(&in_empty[b], ((u >> 1) & 1) ^ 1, wc)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(&in_full[b], 2 * C::kHB);
          load_tile_halves<D, kH64>(smem + C::kOffQh + b * C::kHB, &tmQh, &in_full[b], h * 64, bh);
          load_tile_halves<D, kH64>(smem + C::kOffGh + b * C::kHB, &tmGh, &in_full[b], h * 64, bh);
        }
        ++issued;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int qq = lane + 32 * j;
          put_ext_row(smem + C::kOffBExtS + b * kExt64, qq, nl[j] / c2);
          put_ext_row(smem + C::kOffBExtA + b * kExt64, qq, -de[j]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&in_full[b]);
      }
      if (lane == 0 && *abort_flag) {
        drain_wait_bt(kv_full, 0);
        for (int u = (issued > 2 ? issued - 2 : 0); u < issued; ++u) drain_wait_bt(&in_full[u & 1], (u >> 1) & 1);
      }
    } else if (warp == 5) {
      // -------------------------------------------------------- MMA issuer
      // S'(u), dA'(u) into the slot, then the products of half tile u - 1:
      // dV += r^T Gs and dK1 += u^T Q (r^T, u^T: K-major A operands, 16
      // queries = 32 bytes per K step; G and Q of buffer bp as MN-major B, 16
      // queries = 2 KB per K step, the two 64-column halves of d = 128 8 KB
      // apart).
      if (lane == 0) {
        constexpr long long kStepKm = 2;                       // K-major: +32 bytes per K step
        constexpr long long kStepMn = 128;                     // MN-major: +16 rows (2 KB) per K step
        const uint32_t idesc_s = idesc_bf16(kTile, 64, false, false);
        const uint32_t idesc_acc = idesc_bf16(kTile, D, false, true);
        const uint64_t dK = kdesc(sK, 0), dV = kdesc(sV, 0);
        const uint64_t dAExt = smem_desc_noswizzle(smem_u32(sAExt), 128, 256);
        bool ok = mbar_wait(kv_full, 0, wc);
        if (ok) tc_fence_after();
        for (int u = 0; ok && u <= n; ++u) {
          if (u < n) {
            const int b = u & 1;
            if (!mbar_wait(&in_full[b], (u >> 1) & 1, wc) || !mbar_wait(s_free, (u & 1) ^ 1, wc)) break;
            tc_fence_after();
            const uint64_t dQh = kdesc(smem + C::kOffQh + b * C::kHB, 0);
            const uint64_t dGh = kdesc(smem + C::kOffGh + b * C::kHB, 0);
            const uint64_t dBS = smem_desc_noswizzle(smem_u32(smem + C::kOffBExtS + b * kExt64), 128, 256);
            const uint64_t dBA = smem_desc_noswizzle(smem_u32(smem + C::kOffBExtA + b * kExt64), 128, 256);
            mma_over_d<D>(tmem, dK, kH128, dQh, kH64, idesc_s);
            mma_bf16_at<0, 0>(tmem, dAExt, dBS, idesc_s, 1u);
            mma_over_d<D>(tmem + 64, dV, kH128, dGh, kH64, idesc_s);
            mma_bf16_at<0, 0>(tmem + 64, dAExt, dBA, idesc_s, 1u);
            mma_commit(s_full);
          }
          if (u >= 1) {
            const int up = u - 1, bp = up & 1;
            if (!mbar_wait(x_full, up & 1, wc)) break;
            tc_fence_after();
            const uint64_t dGmn = smem_desc(smem_u32(smem + C::kOffGh + bp * C::kHB), kH64, 1024);
            const uint64_t dQmn = smem_desc(smem_u32(smem + C::kOffQh + bp * C::kHB), kH64, 1024);
            MmaRun<0, 4, kStepKm, kStepMn, false>::go(tmem + C::kTmemAcc0, kdesc(sAT, 0), dGmn, idesc_acc,
                                                      up > 0 ? 1u : 0u);
            MmaRun<0, 4, kStepKm, kStepMn, false>::go(tmem + C::kTmemAcc1, kdesc(sUT, 0), dQmn, idesc_acc,
                                                      up > 0 ? 1u : 0u);
            mma_commit(x_free);
            mma_commit(&in_empty[bp]);
            if (u == n) mma_commit(fin);
          }
        }
        mma_commit(drain);
        drain_wait_bt(drain, 0);
      }
    }
  } else {
    // ------------------------------------------------------ key threads
    if constexpr (RevRegs<D>::kSplit) setmaxnreg_inc<RevRegs<D>::kKey>();
    const int row = warp * 32 + lane;
    const int key = kt * kTile + row;
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
    const int swz = row & 7;
    uint8_t *at_row = sAT + (row >> 3) * 1024 + (row & 7) * 128;
    uint8_t *ut_row = sUT + (row >> 3) * 1024 + (row & 7) * 128;
    float *xp = reinterpret_cast<float *>(smem + C::kOffXp) + warp * 32 * 36;   // d = 128 only
    float grev = 0.f;   // sum of dC over the queries after the current one
    // Checkpoints are read one half tile ahead: they come from DRAM and are
    // needed at the start of each chunk.
    auto ck_of = [&](int uu, int c) { return ((size_t)bh * NC + (half_of(uu) * 2 + c)) * Tp + key; };
    float cpe_n[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) cpe_n[c] = __ldg(cchk + ck_of(0, c));
    bool ok = true;
    for (int u = 0; ok && u < n; ++u) {
      const int b = u & 1, h = half_of(u);
      const float cpe_c[2] = {cpe_n[0], cpe_n[1]};
      if (u + 1 < n) {
#pragma unroll
        for (int c = 0; c < 2; ++c) cpe_n[c] = __ldg(cchk + ck_of(u + 1, c));
      }
      const int q0h = h * 64;
      const bool need_mask = kt * kTile + kTile - 1 > q0h;
      const int row_eff = key - q0h;
      if (!warp_wait(s_full, u & 1, wc)) break;
      tc_fence_after();
      // partial rho buffer b read
      if (!warp_wait(&r_free[b], ((u >> 1) & 1) ^ 1, wc)) break;
      // The two chunks unrolled: at d = 64 the key warps' registers leave the
      // room (backward 13.71 -> 12.84 ms).  Loading both chunks from TMEM at
      // once (one wait, the slot back before any arithmetic) measured slower
      // (12.75 vs 12.46 ms).
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 1 - cc;   // the chunks backwards
        float P[32], A[32], E[32];
        uint32_t at[16];
        tmem_ld32(tmem + lanes + 32 * c, P);
        tmem_ld32(tmem + 64 + lanes + 32 * c, A);
        tmem_wait_ld_r(P);
        tmem_wait_ld_r(A);
        if (cc == 1) release_bt(s_free, lane);
        const size_t ck = ((size_t)bh * NC + (q0h / 32 + c)) * Tp + key;
        const float cpe = cpe_c[c];
        if (need_mask) bwd_chunk_fwd<true, EARLIER, true>(P, A, E, at, row_eff, 32 * c, c2, cpe);
        else bwd_chunk_fwd<false, EARLIER, true>(P, A, E, at, row_eff, 32 * c, c2, cpe);
        gchk[ck] = grev;   // sum of dC after the chunk
        bwd_chunk_rev<EARLIER>(A, E, grev);
        uint32_t ut[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {   // u = p dp
          const float2 x = fmul2(make_float2(P[i], P[i + 1]), make_float2(A[i], A[i + 1]));
          if constexpr (C::kXp) {
            P[i] = x.x;
            P[i + 1] = x.y;
          }
          ut[i / 2] = pack_bf16x2(x.x, x.y);
        }
        // the previous half tile's products must be done reading A^T, u^T
        // (checked once the first chunk is formed, so they run meanwhile)
        if (cc == 0 && !warp_wait(x_free, (u & 1) ^ 1, wc)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int piece = (4 * c + j) ^ swz;
          *reinterpret_cast<uint4 *>(at_row + piece * 16) = make_uint4(at[4 * j], at[4 * j + 1], at[4 * j + 2], at[4 * j + 3]);
          *reinterpret_cast<uint4 *>(ut_row + piece * 16) = make_uint4(ut[4 * j], ut[4 * j + 1], ut[4 * j + 2], ut[4 * j + 3]);
        }
        if constexpr (C::kXp) sRed[(b * 4 + warp) * 64 + 32 * c + lane] = warp_column_sum(P, xp, lane);
      }
      if (!ok) break;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(x_full);
        mbar_arrive(&in_empty[b]);
      }
      if constexpr (!C::kXp) {
        // the warp's partial rho from its u^T rows (the products read them
        // meanwhile)
        *reinterpret_cast<float2 *>(sRed + (b * 4 + warp) * 64 + 2 * lane) = ut_column_sums(sUT + warp * 4096, lane);
        __syncwarp();
      }
      if (lane == 0) mbar_arrive(&r_full[b]);
      // warps 0 and 1 add the four warps' partial sums of the half tile's
      // 64 queries into rho (one atomic per query and key tile)
      if (warp < 2) {
        if (!warp_wait(&r_full[b], (u >> 1) & 1, wc)) {
          ok = false;
          break;
        }
        const int qq = warp * 32 + lane;
        const float *rd = sRed + b * 4 * 64 + qq;
        const float sum = (rd[0] + rd[64]) + (rd[128] + rd[192]);
        if (q0h + qq < T) atomicAdd(rho + (size_t)bh * Tp + q0h + qq, sum);
        __syncwarp();
        if (lane == 0) mbar_arrive(&r_free[b]);
      }
    }
    if (ok && __all_sync(0xffffffffu, !*abort_flag) && warp_wait(fin, 0, wc)) {
      tc_fence_after();
      // dV (TMEM columns 128 ..) of this key out in bf16; dK1 (128 + d ..) in
      // fp32 for the pass that completes dK
      // (tcgen05.ld is warp-collective: every lane loads, only keys < T store)
      float x[32];
#pragma unroll
      for (int part = 0; part < D / 16; ++part) {   // d / 32 parts of dV, then of dK1
        tmem_ld32(tmem + C::kTmemAcc0 + lanes + 32 * part, x);
        tmem_wait_ld_r(x);
        if (key < T) {
          const int col = 32 * (part % (D / 32));
          if (part < D / 32) {
            __nv_bfloat16 *dst = dv + ((size_t)bh * T + key) * D + col;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              reinterpret_cast<uint4 *>(dst)[j] =
                  make_uint4(pack_bf16x2(x[8 * j], x[8 * j + 1]), pack_bf16x2(x[8 * j + 2], x[8 * j + 3]),
                             pack_bf16x2(x[8 * j + 4], x[8 * j + 5]), pack_bf16x2(x[8 * j + 6], x[8 * j + 7]));
          } else {
            float4 *dst = reinterpret_cast<float4 *>(dk1 + ((size_t)bh * T + key) * D + col);
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// L: dK2 = sum_j p_jk rho_j q_j, then dK = c (dK1 - dK2).  Half tiles in
// forward order; one S' slot (the key threads read both chunks at once and
// hand it back), (p rho)^T buffers double-buffered.  (Carrying |rho| in the
// exponent, with sign(rho) q as the operand, saves the product by rho per
// pair but needs a sign-flip pass over Q: backward 11.42 -> 11.49 ms.)
template <int D>
__global__ void __launch_bounds__(kBtThreads, KeyCfg<kModeDk2, D>::kCtasPerSm)
    bwdtc_dk2_kernel(const __grid_constant__ CUtensorMap tmQh, const __grid_constant__ CUtensorMap tmK,
                     const float *__restrict__ nlse2, const float *__restrict__ rho, const float *__restrict__ dk1,
                     __nv_bfloat16 *__restrict__ dk, int BH, int T, int Tp, HeadScale hs, float c_scalar,
                     int *status) {
  using C = KeyCfg<kModeDk2, D>;
  extern __shared__ uint8_t bt_smem_raw[];
  uint8_t *smem = bt_smem_raw + ((1024u - (smem_u32(bt_smem_raw) & 1023u)) & 1023u);
  uint8_t *sK = smem + C::kOffK;
  uint8_t *sAExt = smem + C::kOffAExt;
  float *sRho = reinterpret_cast<float *>(smem + C::kOffRows);
  uint8_t *sPT = smem + C::kOffOp;   // [2] (p rho)^T, K-major
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *k_full = bars;
  uint64_t *in_full = bars + 1;      // [2] half tile b loaded and its rows written
  uint64_t *in_empty = bars + 3;     // [2] its products done and its rows read
  uint64_t *s_full = bars + 5;       // S' slot
  uint64_t *s_free = bars + 7;
  uint64_t *x_full = bars + 9;       // [2] (p rho)^T written
  uint64_t *x_free = bars + 11;      // [2] its product done
  uint64_t *fin = bars + 13;
  uint64_t *drain = bars + 14;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 15);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const TileWork tw = bwd_work(blockIdx.x, BH, T, D, kBwdDk2);
  const int bh = tw.bh, kt = tw.q_tile0;
  const int NH = Tp / 64, hq0 = 2 * kt, n = NH - hq0;
  const float c2 = fmaxf(head_c2(hs, bh, nullptr), 1e-30f);

  if (threadIdx.x == 0) {
    mbar_init(k_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&in_full[b], 2);
      mbar_init(&in_empty[b], 5);   // the issuer's commit + the four key warps
      mbar_init(&x_full[b], 4);
      mbar_init(&x_free[b], 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(fin, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  fill_ones_ext(sAExt, threadIdx.x, kBtThreads);
  zero_smem(smem + C::kOffBExtS, 2 * kExt64, threadIdx.x, kBtThreads);
  fence_proxy_async_smem();
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, status};

  if (warp == 4) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tmQh);
      prefetch_tmap(&tmK);
      mbar_arrive_expect_tx(k_full, C::kTB);
      load_tile_halves<D, kH128>(sK, &tmK, k_full, kt * kTile, bh);
    }
    int issued = 0;
    for (int u = 0; u < n; ++u) {
      const int b = u & 1, h = hq0 + u;
      float nl[2], rh[2];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const size_t idx = (size_t)bh * Tp + h * 64 + lane + 32 * j;
        nl[j] = __ldg(nlse2 + idx);
        rh[j] = __ldg(rho + idx);
      }
      if (!mbar_wait(&in_empty[b], ((u >> 1) & 1) ^ 1, wc)) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&in_full[b], C::kHB);
        load_tile_halves<D, kH64>(smem + C::kOffQh + b * C::kHB, &tmQh, &in_full[b], h * 64, bh);
      }
      ++issued;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int qq = lane + 32 * j;
        put_ext_row(smem + C::kOffBExtS + b * kExt64, qq, nl[j] / c2);
        sRho[b * 64 + qq] = rh[j];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&in_full[b]);
    }
    if (lane == 0 && *abort_flag) {
      drain_wait_bt(k_full, 0);
      for (int u = (issued > 2 ? issued - 2 : 0); u < issued; ++u) drain_wait_bt(&in_full[u & 1], (u >> 1) & 1);
    }
  } else if (warp == 5) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr long long kStepKm = 2, kStepMn = 128;
      const uint32_t idesc_s = idesc_bf16(kTile, 64, false, false);
      const uint32_t idesc_acc = idesc_bf16(kTile, D, false, true);
      const uint64_t dK = kdesc(sK, 0);
      const uint64_t dAExt = smem_desc_noswizzle(smem_u32(sAExt), 128, 256);
      bool ok = mbar_wait(k_full, 0, wc);
      if (ok) tc_fence_after();
      for (int u = 0; ok && u <= n; ++u) {
        if (u < n) {
          const int b = u & 1;
          if (!mbar_wait(&in_full[b], (u >> 1) & 1, wc) || !mbar_wait(s_free, (u & 1) ^ 1, wc)) break;
          tc_fence_after();
          const uint64_t dQh = kdesc(smem + C::kOffQh + b * C::kHB, 0);
          const uint64_t dBS = smem_desc_noswizzle(smem_u32(smem + C::kOffBExtS + b * kExt64), 128, 256);
          mma_over_d<D>(tmem, dK, kH128, dQh, kH64, idesc_s);
          mma_bf16_at<0, 0>(tmem, dAExt, dBS, idesc_s, 1u);
          mma_commit(s_full);
        }
        if (u >= 1) {
          const int up = u - 1, bp = up & 1;
          if (!mbar_wait(&x_full[bp], (up >> 1) & 1, wc)) break;
          tc_fence_after();
          const uint64_t dQmn = smem_desc(smem_u32(smem + C::kOffQh + bp * C::kHB), kH64, 1024);
          MmaRun<0, 4, kStepKm, kStepMn, false>::go(tmem + C::kTmemAcc0, kdesc(sPT + bp * kH128, 0), dQmn,
                                                    idesc_acc, up > 0 ? 1u : 0u);
          mma_commit(&x_free[bp]);
          mma_commit(&in_empty[bp]);
          if (u == n) mma_commit(fin);
        }
      }
      mma_commit(drain);
      drain_wait_bt(drain, 0);
    }
  } else {
    // ------------------------------------------------------ key threads
    const int row = warp * 32 + lane;
    const int key = kt * kTile + row;
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
    const int swz = row & 7;
    const float2 c2v = make_float2(c2, c2);
    bool ok = true;
    for (int u = 0; ok && u < n; ++u) {
      const int b = u & 1, h = hq0 + u;
      const int q0h = h * 64;
      const bool need_mask = kt * kTile + kTile - 1 > q0h;
      const int row_eff = key - q0h;
      uint8_t *pt_row = sPT + b * kH128 + (row >> 3) * 1024 + (row & 7) * 128;
      if (!warp_wait(s_full, u & 1, wc) || !warp_wait(&x_free[b], ((u >> 1) & 1) ^ 1, wc)) break;
      tc_fence_after();
      float P0[32], P1[32];
      tmem_ld32(tmem + lanes, P0);
      tmem_ld32(tmem + lanes + 32, P1);
      tmem_wait_ld_r(P0);
      tmem_wait_ld_r(P1);
      release_bt(s_free, lane);
      const float *rq = sRho + b * 64;
      auto chunk = [&](float (&P)[32], int c) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const float2 x = fmul2(make_float2(P[i], P[i + 1]), c2v);
          float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
          if (need_mask) {
            if (row_eff > 32 * c + i) p0 = 0.f;
            if (row_eff > 32 * c + i + 1) p1 = 0.f;
          }
          const float2 r2 = *reinterpret_cast<const float2 *>(rq + 32 * c + i);
          const float2 pr = fmul2(make_float2(p0, p1), r2);
          pk[i / 2] = pack_bf16x2(pr.x, pr.y);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j)
          *reinterpret_cast<uint4 *>(pt_row + (((4 * c + j) ^ swz) * 16)) =
              make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
      };
      chunk(P0, 0);
      chunk(P1, 1);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&x_full[b]);
        mbar_arrive(&in_empty[b]);
      }
    }
    if (ok && __all_sync(0xffffffffu, !*abort_flag) && warp_wait(fin, 0, wc)) {
      tc_fence_after();
      // dK = c (dK1 - dK2) of this key, out in bf16
      const float cs = hs.tau_bh == nullptr ? c_scalar : c2 * 0.69314718055994531f;
      float x[32];
#pragma unroll
      for (int part = 0; part < D / 32; ++part) {
        tmem_ld32(tmem + C::kTmemAcc0 + lanes + 32 * part, x);
        tmem_wait_ld_r(x);
        if (key < T) {
          const float4 *src = reinterpret_cast<const float4 *>(dk1 + ((size_t)bh * T + key) * D + 32 * part);
          __nv_bfloat16 *dst = dk + ((size_t)bh * T + key) * D + 32 * part;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 a0 = __ldg(src + 2 * j), a1 = __ldg(src + 2 * j + 1);
            reinterpret_cast<uint4 *>(dst)[j] =
                make_uint4(pack_bf16x2((a0.x - x[8 * j]) * cs, (a0.y - x[8 * j + 1]) * cs),
                           pack_bf16x2((a0.z - x[8 * j + 2]) * cs, (a0.w - x[8 * j + 3]) * cs),
                           pack_bf16x2((a1.x - x[8 * j + 4]) * cs, (a1.y - x[8 * j + 5]) * cs),
                           pack_bf16x2((a1.z - x[8 * j + 6]) * cs, (a1.w - x[8 * j + 7]) * cs));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------ query-major pass
// One CTA per (head, 128-query tile), two per SM, walking the key tiles up to
// the diagonal.  Per key tile: S and dA' for the two 64-query halves (one
// TMEM slot pair, reused), one thread per key writing ds (MN-major, the
// layout of the forward's share^T), then dQ += ds K (M = 128 queries, N = 64,
// K = 128 keys) accumulating in TMEM.
template <int D>
struct QCfg {
  static constexpr uint32_t kTB = kTile * D * 2;
  // two key-tile buffers (tile u in buffer u % 2), one value tile, and ds of
  // one 64-query half (16 key groups x 1 KB)
  static constexpr uint32_t kOffQ = 0, kOffG = kTB, kOffK = 2 * kTB, kOffV = 4 * kTB;
  static constexpr uint32_t kOffDs = 5 * kTB;
  static constexpr uint32_t kOffAExt = kOffDs + 16 * 1024;
  static constexpr uint32_t kOffBExtS = kOffAExt + kExt128;       // 128 query rows
  static constexpr uint32_t kOffBExtA = kOffBExtS + kExt128;
  static constexpr uint32_t kOffRho = kOffBExtA + kExt128;        // [128] fp32, negated
  static constexpr uint32_t kOffBar = kOffRho + 128 * 4;
  static constexpr int kSmemBytes = kOffBar + 256 + 1024;
  static constexpr int kCtasPerSm = D == 64 ? 2 : 1;
  // TMEM: S' (64 columns), dA' (64), then dQ as two M = 64 accumulators
  // (queries 0..63 and 64..127 of the tile), d columns each
  static constexpr uint32_t kTmemDQ = 128;
  static constexpr uint32_t kTmemCols = D == 64 ? 256 : 512;
  static_assert(kSmemBytes <= 232448, "shared memory");
};

template <int D, bool EARLIER>
__global__ void __launch_bounds__(kBtThreads, QCfg<D>::kCtasPerSm)
    bwdtc_q_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmG,
                   const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                   const float *__restrict__ nlse2, const float *__restrict__ delta, const float *__restrict__ rho, const float *__restrict__ cchk, const float *__restrict__ gchk,
                   __nv_bfloat16 *__restrict__ dq, int BH, int T, int Tp, HeadScale hs, float c_scalar,
                   int *status) {
  using C = QCfg<D>;
  extern __shared__ uint8_t bt_smem_raw[];
  uint8_t *smem = bt_smem_raw + ((1024u - (smem_u32(bt_smem_raw) & 1023u)) & 1023u);
  uint8_t *sQ = smem + C::kOffQ, *sG = smem + C::kOffG, *sK = smem + C::kOffK, *sV = smem + C::kOffV;
  uint8_t *sDs = smem + C::kOffDs, *sAExt = smem + C::kOffAExt;
  uint8_t *sBExtS = smem + C::kOffBExtS, *sBExtA = smem + C::kOffBExtA;
  float *sRho = reinterpret_cast<float *>(smem + C::kOffRho);
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::kOffBar);
  uint64_t *q_full = bars;           // Q, G tiles and the query rows
  uint64_t *k_full = bars + 1, *k_empty = bars + 3;   // [2]: key buffer u % 2
  uint64_t *v_full = bars + 5, *v_empty = bars + 6;
  uint64_t *s_full = bars + 7, *s_free = bars + 8;
  uint64_t *ds_full = bars + 9, *ds_free = bars + 10;   // per step it = 2 u + half
  uint64_t *fin = bars + 11, *drain = bars + 12;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 13);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int NC = Tp / 32;
  const TileWork tw = bwd_work(blockIdx.x, BH, T, D, kBwdDq);
  const int bh = tw.bh, qt = tw.q_tile0;
  const int n = qt + 1;                                              // key tiles 0 .. qt
  const float c2 = fmaxf(head_c2(hs, bh, nullptr), 1e-30f);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 2);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&k_full[i], 1);
      mbar_init(&k_empty[i], 1);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    mbar_init(s_full, 1);
    mbar_init(s_free, 4);
    mbar_init(ds_full, 4);
    mbar_init(ds_free, 1);
    mbar_init(fin, 1);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  fill_ones_ext(sAExt, threadIdx.x, kBtThreads);
  zero_smem(sBExtS, 2 * kExt128, threadIdx.x, kBtThreads);   // both extension row blocks
  fence_proxy_async_smem();
  if (warp == 5) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const WaitCtx wc{abort_flag, status};

  if (warp == 4) {
    // ---------------------------------------------------------- producer
    if (lane == 0) {
      prefetch_tmap(&tmQ);
      prefetch_tmap(&tmG);
      prefetch_tmap(&tmK);
      prefetch_tmap(&tmV);
      mbar_arrive_expect_tx(q_full, 2 * C::kTB);
      load_tile_halves<D, kH128>(sQ, &tmQ, q_full, qt * kTile, bh);
      load_tile_halves<D, kH128>(sG, &tmG, q_full, qt * kTile, bh);
    }
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int qq = lane + 32 * j;
      const size_t idx = (size_t)bh * Tp + qt * kTile + qq;
      put_ext_row(sBExtS, qq, __ldg(nlse2 + idx) / c2);
      put_ext_row(sBExtA, qq, -__ldg(delta + idx));
      sRho[qq] = -rho[idx];   // negated: ds = p (dp + (-rho)) on the packed pipe
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(q_full);
    int issued = 0;
    if (lane == 0) {
      for (int u = 0; u < n; ++u) {
        const int kb = u & 1;
        if (!mbar_wait(&k_empty[kb], ((u >> 1) & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(&k_full[kb], C::kTB);
        load_tile_halves<D, kH128>(sK + kb * C::kTB, &tmK, &k_full[kb], u * kTile, bh);
        if (!mbar_wait(v_empty, (u & 1) ^ 1, wc)) break;
        mbar_arrive_expect_tx(v_full, C::kTB);
        load_tile_halves<D, kH128>(sV, &tmV, v_full, u * kTile, bh);
        ++issued;
      }
      if (*abort_flag) {
        drain_wait_bt(q_full, 0);
        for (int u = (issued > 2 ? issued - 2 : 0); u <= issued && u < n; ++u)   // key loads possibly in flight
          drain_wait_bt(&k_full[u & 1], (u >> 1) & 1);
        if (issued > 0) drain_wait_bt(v_full, (issued - 1) & 1);
      }
    }
  } else if (warp == 5) {
    // -------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr long long kStepMn = 128;
      const uint32_t idesc_s = idesc_bf16(kTile, 64, false, false);
      const uint32_t idesc_q = idesc_bf16(64, D, true, true);   // one 64-query half: M = 64
      const uint64_t dV = kdesc(sV, 0);
      const uint64_t dAExt = smem_desc_noswizzle(smem_u32(sAExt), 128, 256);
      // ds: MN-major, one 64-query block, 8-key groups 1 KB apart (SBO); K as
      // the MN-major B operand (16 keys = 2 KB per K step, its 64-column
      // halves 16 KB apart)
      const uint64_t dDs = smem_desc(smem_u32(sDs), 16384, 1024);
      // Steps it = 2 u + hh (key tile u, query half hh).  The events of the
      // key threads come in the order: slot of step it released (its S' and
      // dA' loaded), ds of step it written, slot of step it + 1 released ...;
      // so the issuer walks S(0), S(1), dQ(0), S(2), dQ(1), ... with blocking
      // waits.  dQ(it) adds ds K(u) into the half's accumulator; key tile u's
      // buffer goes back to the producer after dQ(2 u + 1), so tile u + 1
      // (the other buffer) has been loading all along.
      auto issue_s = [&](int it) -> bool {
        const int u = it >> 1, hh = it & 1;
        if (hh == 0 && (!mbar_wait(&k_full[u & 1], (u >> 1) & 1, wc) || !mbar_wait(v_full, u & 1, wc)))
          return false;
        if (!mbar_wait(s_free, (it & 1) ^ 1, wc)) return false;
        tc_fence_after();
        // the query half: rows 64 hh.. of the Q / G tiles (8 KB on) and of
        // the extension rows (8 groups of 256 bytes on)
        const uint64_t dK = kdesc(sK + (u & 1) * C::kTB, 0);
        const uint64_t dQh = kdesc(sQ + hh * 8192, 0), dGh = kdesc(sG + hh * 8192, 0);
        const uint64_t dBS = smem_desc_noswizzle(smem_u32(sBExtS) + hh * 2048, 128, 256);
        const uint64_t dBA = smem_desc_noswizzle(smem_u32(sBExtA) + hh * 2048, 128, 256);
        mma_over_d<D>(tmem, dK, kH128, dQh, kH128, idesc_s);
        mma_bf16_at<0, 0>(tmem, dAExt, dBS, idesc_s, 1u);
        mma_over_d<D>(tmem + 64, dV, kH128, dGh, kH128, idesc_s);
        mma_bf16_at<0, 0>(tmem + 64, dAExt, dBA, idesc_s, 1u);
        mma_commit(s_full);
        if (hh == 1) mma_commit(v_empty);
        return true;
      };
      auto issue_dq = [&](int it) -> bool {
        const int u = it >> 1, hh = it & 1;
        if (!mbar_wait(ds_full, it & 1, wc)) return false;
        tc_fence_after();
        const uint64_t dKmn = smem_desc(smem_u32(sK + (u & 1) * C::kTB), kH128, 1024);
        MmaRun<0, kTile / 16, kStepMn, kStepMn, false>::go(tmem + C::kTmemDQ + hh * D, dDs, dKmn, idesc_q,
                                                          u > 0 ? 1u : 0u);
        mma_commit(ds_free);
        if (hh == 1) mma_commit(&k_empty[u & 1]);
        if (it == 2 * n - 1) mma_commit(fin);
        return true;
      };
      bool ok = mbar_wait(q_full, 0, wc);
      if (ok) tc_fence_after();
      ok = ok && issue_s(0);
      for (int it = 0; ok && it < 2 * n; ++it) {
        if (it + 1 < 2 * n && !issue_s(it + 1)) break;
        if (!issue_dq(it)) break;
      }
      mma_commit(drain);
      drain_wait_bt(drain, 0);
    }
  } else {
    // ------------------------------------------------------ key threads
    const int row = warp * 32 + lane;   // key row of the current key tile
    const uint32_t lanes = (uint32_t)(warp * 32) << 16;
    const int swz = row & 7;
    uint8_t *ds_row = sDs + (row >> 3) * 1024 + (row & 7) * 128;
    bool ok = warp_wait(q_full, 0, wc);
    // checkpoints of step it = 2 u + hh (key tile u, query half hh), read one
    // step ahead
    auto ck_of = [&](int it, int c) {
      return ((size_t)bh * NC + (qt * kTile + 64 * (it & 1) + 32 * c) / 32) * Tp + (it >> 1) * kTile + row;
    };
    float cpe_n[2], g_n[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      cpe_n[c] = __ldg(cchk + ck_of(0, c));
      g_n[c] = __ldg(gchk + ck_of(0, c));
    }
    for (int u = 0; ok && u < n; ++u) {
      const bool diag = u == qt;          // keys after queries only on the diagonal tile
      for (int hh = 0; hh < 2 && ok; ++hh) {
        const int it = 2 * u + hh;
        const float cpe_c[2] = {cpe_n[0], cpe_n[1]};
        const float g_c[2] = {g_n[0], g_n[1]};
        if (it + 1 < 2 * n) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            cpe_n[c] = __ldg(cchk + ck_of(it + 1, c));
            g_n[c] = __ldg(gchk + ck_of(it + 1, c));
          }
        }
        if (!warp_wait(s_full, it & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int c = 0; c < 2; ++c) {
          float P[32], A[32], E[32];
          uint32_t at[16];
          tmem_ld32(tmem + lanes + 32 * c, P);
          tmem_ld32(tmem + 64 + lanes + 32 * c, A);
          tmem_wait_ld_r(P);
          tmem_wait_ld_r(A);
          if (c == 1) release_bt(s_free, lane);
          const int col0 = 64 * hh + 32 * c;   // first query of the chunk inside the tile
          const float cpe = cpe_c[c];
          if (diag) bwd_chunk_fwd<true, EARLIER, false>(P, A, E, at, row, col0, c2, cpe);
          else bwd_chunk_fwd<false, EARLIER, false>(P, A, E, at, row, col0, c2, cpe);
          float g0 = g_c[c];
          bwd_chunk_rev<EARLIER>(A, E, g0);
          uint32_t ds[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {   // ds = p (dp - rho)
            const float2 r2 = *reinterpret_cast<const float2 *>(sRho + col0 + 2 * i);
            const float2 x = fmul2(make_float2(P[2 * i], P[2 * i + 1]),
                                   fadd2(make_float2(A[2 * i], A[2 * i + 1]), r2));
            ds[i] = pack_bf16x2(x.x, x.y);
          }
          // the previous step's dQ product must be done reading the ds buffer
          if (c == 0 && !warp_wait(ds_free, (it & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          // 32 queries of chunk c of this half -> 16-byte pieces c * 4 .. + 3
          // of this key's 128-byte row of the half's ds block, swizzled
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4 *>(ds_row + (((c * 4 + j) ^ swz) * 16)) =
                make_uint4(ds[4 * j], ds[4 * j + 1], ds[4 * j + 2], ds[4 * j + 3]);
        }
        if (!ok) break;
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(ds_full);
      }
    }
    if (ok && __all_sync(0xffffffffu, !*abort_flag) && warp_wait(fin, 0, wc)) {
      tc_fence_after();
      // dQ rows: an M = 64 accumulator keeps row m on TMEM lane
      // (m / 16) * 32 + m % 16, so lane l < 16 of warp w holds row 16 w + l
      // of each half's accumulator
      const float cs = hs.tau_bh == nullptr ? c_scalar : c2 * 0.69314718055994531f;
      float x[32];
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int qi = qt * kTile + 64 * hh + 16 * warp + lane;
#pragma unroll
        for (int part = 0; part < D / 32; ++part) {
          tmem_ld32(tmem + C::kTmemDQ + hh * D + lanes + 32 * part, x);
          tmem_wait_ld_r(x);
          if (lane < 16 && qi < T) {
            __nv_bfloat16 *dst = dq + ((size_t)bh * T + qi) * D + 32 * part;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              reinterpret_cast<uint4 *>(dst)[j] =
                  make_uint4(pack_bf16x2(x[8 * j] * cs, x[8 * j + 1] * cs), pack_bf16x2(x[8 * j + 2] * cs, x[8 * j + 3] * cs),
                             pack_bf16x2(x[8 * j + 4] * cs, x[8 * j + 5] * cs), pack_bf16x2(x[8 * j + 6] * cs, x[8 * j + 7] * cs));
          }
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ------------------------------------------------------------------- host
bool make_bf16_tile_map(CUtensorMap *m, const void *base, int BH, int T, int d, int rows);
int launch_sweep_bf16_chk(const void *q, const void *k, const void *v, const float *nlse2, float *acc, float *cchk,
                          int BH, int T, int d, HeadScale hs, float eps, bool earlier, int *status,
                          cudaStream_t stream);

template <int D, bool EARLIER>
static int launch_passes(const CUtensorMap *maps, float *nlse2, float *delta, float *rho, float *cchk,
                         float *gchk, float *dk1, void *dq, void *dk, void *dv, int BH, int T, int Tp, HeadScale hs,
                         float c, int *status, cudaStream_t stream) {
  using CR = KeyCfg<kModeRev, D>;
  using CL = KeyCfg<kModeDk2, D>;
  // The shared-memory opt-in is a per-device function attribute.
  static PerDeviceOnce once;
  const int prep = once.run([] {
    if constexpr (RevRegs<D>::kSplit) {
      // the register split must fit what the block is launched with, or the
      // key warps' setmaxnreg.inc would never complete: refuse otherwise
      cudaFuncAttributes fa;
      if (cudaFuncGetAttributes(&fa, bwdtc_rev_kernel<D, EARLIER>) != cudaSuccess) return (int)DA_ERR_CUDA;
      if (fa.numRegs * RevRegs<D>::kThreads < RevRegs<D>::kNeeded || fa.numRegs > RevRegs<D>::kKey ||
          fa.numRegs < RevRegs<D>::kCtl)
        return (int)DA_ERR_UNSUPPORTED;
    }
    return (cudaFuncSetAttribute(bwdtc_rev_kernel<D, EARLIER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CR::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(bwdtc_dk2_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 CL::kSmemBytes) != cudaSuccess ||
            cudaFuncSetAttribute(bwdtc_q_kernel<D, EARLIER>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 QCfg<D>::kSmemBytes) != cudaSuccess)
               ? DA_ERR_CUDA
               : DA_OK;
  });
  if (prep != DA_OK) return prep;
  const int NT = Tp / kTile;
  const unsigned grid = (unsigned)(NT * BH);
  // maps: 0 Q (64-row boxes), 1 dout / R (64), 2 K (128), 3 V (128), 4 Q (128), 5 dout / R (128)
  bwdtc_rev_kernel<D, EARLIER><<<grid, RevRegs<D>::kThreads, CR::kSmemBytes, stream>>>(
      maps[0], maps[1], maps[2], maps[3], nlse2, delta, rho, cchk, gchk, dk1,
      static_cast<__nv_bfloat16 *>(dv), BH, T, Tp, hs, status);
  bwdtc_dk2_kernel<D><<<grid, kBtThreads, CL::kSmemBytes, stream>>>(
      maps[0], maps[2], nlse2, rho, dk1, static_cast<__nv_bfloat16 *>(dk), BH, T, Tp, hs, c, status);
  bwdtc_q_kernel<D, EARLIER><<<grid, kBtThreads, QCfg<D>::kSmemBytes, stream>>>(
      maps[4], maps[5], maps[2], maps[3], nlse2, delta, rho, cchk, gchk, static_cast<__nv_bfloat16 *>(dq),
      BH, T, Tp, hs, c, status);
  return cudaGetLastError() == cudaSuccess ? DA_OK : DA_ERR_CUDA;
}

// The tensor-core backward (bf16, d = 64 or 128): the passes in the file header.
// have_fwd_state: the workspace already holds -lse2, the forward accumulators
// and the demand checkpoints of a forward run for these inputs (the forward
// kept them), so pass F is skipped.
int launch_bwd_bf16_tc(const void *q, const void *k, const void *v, const void *dout, const float *lse2, void *dq,
                       void *dk, void *dv, int BH, int T, int d, HeadScale hs, float c, float eps, bool earlier,
                       bool have_fwd_state, uint8_t *ws, cudaStream_t stream) {
  const BwdTcWorkspace L = bwd_tc_workspace_layout(BH, T, d);
  const int Tp = (int)t_pad(T);
  const int64_t rows = (int64_t)BH * Tp;
  int *status = reinterpret_cast<int *>(ws);
  float *nlse2 = reinterpret_cast<float *>(ws + L.nlse2_off);
  float *acc = reinterpret_cast<float *>(ws + L.acc_off);
  float *delta = reinterpret_cast<float *>(ws + L.rows_off), *rho = delta + rows;
  float *cchk = reinterpret_cast<float *>(ws + L.cchk_off);
  float *gchk = reinterpret_cast<float *>(ws + L.gchk_off);
  float *dk1 = reinterpret_cast<float *>(ws + L.dk1_off);
  __nv_bfloat16 *gs = reinterpret_cast<__nv_bfloat16 *>(ws + L.gs_off);   // dout / R
  CUtensorMap maps[6];
  if (!make_bf16_tile_map(&maps[0], q, BH, T, d, 64) || !make_bf16_tile_map(&maps[1], gs, BH, T, d, 64) ||
      !make_bf16_tile_map(&maps[2], k, BH, T, d, kTile) || !make_bf16_tile_map(&maps[3], v, BH, T, d, kTile) ||
      !make_bf16_tile_map(&maps[4], q, BH, T, d, kTile) || !make_bf16_tile_map(&maps[5], gs, BH, T, d, kTile))
    return DA_ERR_CUDA;
  const unsigned gp = (unsigned)((rows + 255) / 256), gr = (unsigned)((rows * 16 + 255) / 256);
  if (!have_fwd_state) {
    if (d == 128) bwdtc_prep<128><<<gp, 256, 0, stream>>>(lse2, nlse2, acc, BH, T, Tp);
    else bwdtc_prep<64><<<gp, 256, 0, stream>>>(lse2, nlse2, acc, BH, T, Tp);
    const int st = launch_sweep_bf16_chk(q, k, v, nlse2, acc, cchk, BH, T, d, hs, eps, earlier, status, stream);
    if (st != DA_OK) return st;
  }
  const __nv_bfloat16 *g = static_cast<const __nv_bfloat16 *>(dout);
  if (d == 128) bwdtc_rows<128><<<gr, 256, 0, stream>>>(acc, g, gs, delta, rho, BH, T, Tp);
  else bwdtc_rows<64><<<gr, 256, 0, stream>>>(acc, g, gs, delta, rho, BH, T, Tp);
#define DA_BWD_PASSES_ARGS maps, nlse2, delta, rho, cchk, gchk, dk1, dq, dk, dv, BH, T, Tp, hs, c, status, stream
  if (d == 128)
    return earlier ? launch_passes<128, true>(DA_BWD_PASSES_ARGS) : launch_passes<128, false>(DA_BWD_PASSES_ARGS);
  return earlier ? launch_passes<64, true>(DA_BWD_PASSES_ARGS) : launch_passes<64, false>(DA_BWD_PASSES_ARGS);
#undef DA_BWD_PASSES_ARGS
}

}  // namespace da
