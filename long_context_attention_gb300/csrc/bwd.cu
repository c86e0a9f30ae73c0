// Backward of dilution attention: dq, dk, dv of sum(dout * out).
//
// The pages state only that exact gradients exist ("DilutionAttention v0.1.0
// · results", last section); the chain rule through the operator of section
// "The operator" gives, per (batch, head), with c = tau/sqrt(d),
// D_jk = committed_jk + p_jk + eps, r = share, R_j = sum_k r_jk, A = r / R
// (the earlier-demand-only variant: D_jk = committed_jk + eps and the direct
// term of dp_jk is dr_jk / D_jk):
//
//   dV_k   = sum_j A_jk g_j                      (g = dout)
//   dr_jk  = (g_j . v_k - g_j . out_j) / R_j
//   dC_jk  = -dr_jk p_jk / D_jk^2                 (d share / d committed)
//   dp_jk  = dr_jk (committed_jk + eps) / D_jk^2 + sum_{i > j} dC_ik
//   rho_j  = sum_k p_jk dp_jk
//   ds_jk  = p_jk (dp_jk - rho_j)                 (softmax)
//   dQ_j   = c sum_k ds_jk k_k,   dK_k = c sum_j ds_jk q_j
//
// One thread owns one key and walks its column of queries, so the column
// sums are running registers:
//   pass 0 (queries ascending): committed_jk exactly; the column total Dtot_k
//          (fp64), the row sums R_j = sum_k r_jk and Y_j = sum_k r_jk (g_j.v_k),
//          so g_j . out_j = Y_j / R_j (both reduced across keys with fp32
//          atomics).  The backward recomputes these from its own bids rather
//          than taking the forward's rounded outputs.
//   pass 1 (queries descending): committed_jk = Dtot_k - sum_{i >= j} p_ik in
//          fp64 (no cancellation trouble near the diagonal), the reverse sum
//          of dC, dp; rho_j (atomics across key blocks) and dV_k (registers).
//   pass 2 (descending): dp again, ds, dK_k (registers), dQ (shared-memory
//          staging of ds, fp32 atomics across key blocks).
//   bwd_final: dq accumulator -> dq in the output type.
// This is the straightforward SIMT version (fp32 arithmetic for fp32 and
// bf16 inputs), instantiated for d = 64 and d = 128; the tensor-core version
// is future work.
#include "da_internal.h"

#include <cuda_bf16.h>

namespace da {

constexpr int kBwKeys = 128;   // keys per CTA (one per thread)
constexpr int kBwQ = 32;       // queries staged per chunk

template <typename E>
__device__ __forceinline__ float ld_e(const E *p) {
  if constexpr (sizeof(E) == 4) return *p;
  else return __bfloat162float(*p);
}
template <typename E>
__device__ __forceinline__ void st_e(E *p, float x) {
  if constexpr (sizeof(E) == 4) *p = x;
  else *p = __float2bfloat16_rn(x);
}

template <int D>
struct BwdSmem {
  float kT[D][kBwKeys];       // this block's keys, transposed (conflict-free column reads)
  float vT[D][kBwKeys];       // and values
  float q[kBwQ][D];           // query chunk
  float g[kBwQ][D];           // dout chunk
  float lse2[kBwQ], rinv[kBwQ], delta[kBwQ], rho[kBwQ];
  float ds[kBwQ][kBwKeys + 1];
  float red[kBwQ][4];         // per-warp partial sums of rho
};

__global__ void bwd_zero(float *__restrict__ rowbuf, float *__restrict__ dq_acc, int64_t rows, int d) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < rows * 4) rowbuf[i] = 0.f;          // R, Y, rho, (spare)
  if (i < rows * d) dq_acc[i] = 0.f;
}

// Reverse-walk step for one key at query j: with srev = sum_{i > j} p_ik
// (fp64) and grev = sum_{i > j} dC_ik, returns dp_jk and A_jk.
struct ColState {
  double dtot, srev;
  float grev;
};

__device__ __forceinline__ float col_step(ColState &cs, float p, float dA, float delta, float rinv, float eps,
                                          bool earlier, float &a_out) {
  const float cpe = (float)(cs.dtot - cs.srev - (double)p) + eps;   // committed + eps
  const float den = earlier ? cpe : cpe + p;
  const float inv = 1.f / den;
  const float r = p * inv;
  a_out = r * rinv;
  const float dr = (dA - delta) * rinv;
  const float inv2 = inv * inv;
  const float dC = -dr * p * inv2;
  const float dp = (earlier ? dr * inv : dr * cpe * inv2) + cs.grev;
  cs.grev += dC;
  cs.srev += (double)p;
  return dp;
}

template <typename E, int D, int PASS>
__global__ void __launch_bounds__(kBwKeys)
    bwd_pass(const E *__restrict__ q, const E *__restrict__ k, const E *__restrict__ v, const E *__restrict__ g,
             const float *__restrict__ lse2, double *__restrict__ dtot, float *__restrict__ Rsum,
             float *__restrict__ Ysum, float *__restrict__ rho, float *__restrict__ dq_acc, E *__restrict__ dk_out,
             E *__restrict__ dv_out, int T, float c_scalar, HeadScale hs, float eps, bool earlier) {
  extern __shared__ float4 bw_smem_raw[];
  BwdSmem<D> &S = *reinterpret_cast<BwdSmem<D> *>(bw_smem_raw);
  const int bh = blockIdx.y;
  // natural-log scale c = tau / sqrt(d) of this head (c2 = c log2(e))
  const float c2 = head_c2(hs, bh, nullptr);
  const float c = hs.tau_bh == nullptr ? c_scalar : c2 * 0.69314718055994531f;
  const int tid = threadIdx.x, lane = tid % 32, warp = tid / 32;
  const int key0 = blockIdx.x * kBwKeys;
  const int key = key0 + tid;
  const size_t base = (size_t)bh * T;
  for (int e = tid; e < kBwKeys * D; e += kBwKeys) {
    const int kk = e / D, t = e % D;
    const bool ok = key0 + kk < T;
    S.kT[t][kk] = ok ? ld_e(k + (base + key0 + kk) * D + t) : 0.f;
    S.vT[t][kk] = ok ? ld_e(v + (base + key0 + kk) * D + t) : 0.f;
  }
  double csum = 0.0;   // pass 0: committed (sum of earlier bids) of this key
  ColState cs{(PASS > 0 && key < T) ? dtot[base + key] : 0.0, 0.0, 0.f};
  float accv[D];      // dV_k (pass 1) or dK_k / c (pass 2)
#pragma unroll
  for (int t = 0; t < D; ++t) accv[t] = 0.f;
  const int nchunks = (T - key0 + kBwQ - 1) / kBwQ;
  for (int cc = 0; cc < nchunks; ++cc) {
    const int ci = (PASS == 0) ? cc : nchunks - 1 - cc;   // pass 0 ascends, passes 1-2 descend
    const int q0 = key0 + ci * kBwQ;
    __syncthreads();
    for (int e = tid; e < kBwQ * D; e += kBwKeys) {
      const int r = e / D, t = e % D;
      const bool ok = q0 + r < T;
      S.q[r][t] = ok ? ld_e(q + (base + q0 + r) * D + t) : 0.f;
      S.g[r][t] = ok ? ld_e(g + (base + q0 + r) * D + t) : 0.f;
    }
    if (tid < kBwQ) {
      const bool ok = q0 + tid < T;
      S.lse2[tid] = ok ? lse2[base + q0 + tid] : INFINITY;
      if (PASS > 0) {
        const float R = ok ? Rsum[base + q0 + tid] : 1.f;
        S.rinv[tid] = 1.f / R;
        S.delta[tid] = ok ? Ysum[base + q0 + tid] / R : 0.f;   // g_j . out_j
        S.rho[tid] = (PASS == 2 && ok) ? rho[base + q0 + tid] : 0.f;
      }
    }
    __syncthreads();
    for (int rr = 0; rr < kBwQ; ++rr) {
      const int r = (PASS == 0) ? rr : kBwQ - 1 - rr;
      const int j = q0 + r;
      float c0 = 0.f, c1 = 0.f;   // pass 0: r, r dA; pass 1: p dp; pass 2: ds
      if (key < T && key <= j && j < T) {
        float sdot = 0.f, dA = 0.f;
#pragma unroll 16
        for (int t = 0; t < D; ++t) {
          sdot = fmaf(S.q[r][t], S.kT[t][tid], sdot);
          dA = fmaf(S.g[r][t], S.vT[t][tid], dA);
        }
        const float p = exp2f(sdot * c2 - S.lse2[r]);
        if (PASS == 0) {
          const float share = p / ((earlier ? (float)csum : (float)csum + p) + eps);
          csum += (double)p;
          c0 = share;
          c1 = share * dA;
        } else {
          float a;
          const float dp = col_step(cs, p, dA, S.delta[r], S.rinv[r], eps, earlier, a);
          if (PASS == 1) {
            c0 = p * dp;
#pragma unroll
            for (int t = 0; t < D; ++t) accv[t] = fmaf(a, S.g[r][t], accv[t]);
          } else {
            const float ds = p * (dp - S.rho[r]);
            c0 = ds;
#pragma unroll
            for (int t = 0; t < D; ++t) accv[t] = fmaf(ds, S.q[r][t], accv[t]);
          }
        }
      }
      if (PASS < 2) {
        float w0 = c0, w1 = c1;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
          w0 += __shfl_xor_sync(0xffffffffu, w0, off);
          if (PASS == 0) w1 += __shfl_xor_sync(0xffffffffu, w1, off);
        }
        if (lane == 0) {
          S.red[r][warp] = w0;
          if (PASS == 0) S.ds[r][warp] = w1;
        }
      } else {
        S.ds[r][tid] = c0;
      }
    }
    __syncthreads();
    if (PASS < 2) {
      if (tid < kBwQ && q0 + tid < T) {
        const float s0 = S.red[tid][0] + S.red[tid][1] + S.red[tid][2] + S.red[tid][3];
        if (PASS == 0) {
          atomicAdd(Rsum + base + q0 + tid, s0);
          atomicAdd(Ysum + base + q0 + tid, S.ds[tid][0] + S.ds[tid][1] + S.ds[tid][2] + S.ds[tid][3]);
        } else {
          atomicAdd(rho + base + q0 + tid, s0);
        }
      }
    } else {
      // dQ_j += c sum_k ds_jk k_k over this block's keys: thread (group, dim),
      // RG = 128 / d row groups of 32 / RG queries.
      constexpr int RG = kBwKeys / D;
      const int dim = tid % D, half = tid / D;
      for (int rq = 0; rq < kBwQ / RG; ++rq) {
        const int r = half * (kBwQ / RG) + rq;
        if (q0 + r >= T) break;
        float a = 0.f;
        for (int kk = 0; kk < kBwKeys; ++kk) a = fmaf(S.ds[r][kk], S.kT[dim][kk], a);
        atomicAdd(dq_acc + (base + q0 + r) * D + dim, c * a);
      }
    }
  }
  if (key < T) {
    if (PASS == 0) {
      dtot[base + key] = csum;
    } else if (PASS == 1) {
#pragma unroll
      for (int t = 0; t < D; ++t) st_e(dv_out + (base + key) * D + t, accv[t]);
    } else {
#pragma unroll
      for (int t = 0; t < D; ++t) st_e(dk_out + (base + key) * D + t, c * accv[t]);
    }
  }
}

template <typename E>
__global__ void bwd_final(const float *__restrict__ dq_acc, E *__restrict__ dq, int64_t n) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) st_e(dq + i, dq_acc[i]);
}

template <typename E, int D>
static cudaError_t launch_bwd_t(const void *q, const void *k, const void *v, const void *dout, const float *lse2,
                                void *dq, void *dk, void *dv, int BH, int T, float c, HeadScale hs, float eps,
                                bool earlier, double *dtot, float *rowbuf, float *dq_acc, cudaStream_t stream) {
  const int64_t rows = (int64_t)BH * T;
  float *Rsum = rowbuf, *Ysum = rowbuf + rows, *rho = rowbuf + 2 * rows;
  const int64_t nz = rows * D;
  bwd_zero<<<(unsigned)((nz + 255) / 256), 256, 0, stream>>>(rowbuf, dq_acc, rows, D);
  const size_t smem = sizeof(BwdSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(bwd_pass<E, D, 0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_pass<E, D, 1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(bwd_pass<E, D, 2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid((T + kBwKeys - 1) / kBwKeys, BH);
#define DA_BWD_ARGS                                                                                              \
  (const E *)q, (const E *)k, (const E *)v, (const E *)dout, lse2, dtot, Rsum, Ysum, rho, dq_acc, (E *)dk, (E *)dv, T, \
      c, hs, eps, earlier
  bwd_pass<E, D, 0><<<grid, kBwKeys, smem, stream>>>(DA_BWD_ARGS);
  bwd_pass<E, D, 1><<<grid, kBwKeys, smem, stream>>>(DA_BWD_ARGS);
  bwd_pass<E, D, 2><<<grid, kBwKeys, smem, stream>>>(DA_BWD_ARGS);
#undef DA_BWD_ARGS
  bwd_final<E><<<(unsigned)((nz + 255) / 256), 256, 0, stream>>>(dq_acc, (E *)dq, nz);
  return cudaGetLastError();
}

cudaError_t launch_bwd(const void *q, const void *k, const void *v, const void *dout, const float *lse2, void *dq,
                       void *dk, void *dv, int BH, int T, int d, float c, HeadScale hs, float eps, bool earlier,
                       int dtype, double *dtot, float *rowbuf, float *dq_acc, cudaStream_t stream) {
#define DA_BWD_LAUNCH_ARGS q, k, v, dout, lse2, dq, dk, dv, BH, T, c, hs, eps, earlier, dtot, rowbuf, dq_acc, stream
  if (dtype == DA_BF16)
    return d == 128 ? launch_bwd_t<__nv_bfloat16, 128>(DA_BWD_LAUNCH_ARGS)
                    : launch_bwd_t<__nv_bfloat16, 64>(DA_BWD_LAUNCH_ARGS);
  return d == 128 ? launch_bwd_t<float, 128>(DA_BWD_LAUNCH_ARGS) : launch_bwd_t<float, 64>(DA_BWD_LAUNCH_ARGS);
#undef DA_BWD_LAUNCH_ARGS
}

}  // namespace da
