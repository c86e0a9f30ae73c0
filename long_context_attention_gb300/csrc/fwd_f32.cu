// fp32 SIMT forward of dilution attention: the correctness anchor.
//
// Three steps per (batch, head), "DilutionAttention v0.1.0 · results",
// section "The operator":
//   1. f32_rowstats: the causal-softmax normaliser of every query row,
//      lse2_i = log2 sum_{k<=i} 2^(x_ik), x = s * tau/sqrt(d) * log2(e), kept
//      as the row max m_i and log2 of the max-shifted sum.
//   2. f32_sweep: one CTA per 128 keys, one thread per key.  Walking the
//      queries in causal order, each thread keeps its key's demand from
//      earlier queries (the exclusive column cumsum) in a register:
//      p = 2^(x - lse2), share = p / (committed + p + eps), committed += p
//      (Kahan-compensated); the earlier-demand-only variant divides by
//      committed + eps.
//      The shares of 32 queries are staged in shared memory and multiplied
//      by the CTA's 128 value rows; the partial numerators and share row
//      sums are added (fp32 atomics) into the accumulator acc[row][0..64].
//   3. finalize (shared with the bf16 path): out = acc[0:d] / acc[d].
// No tensor cores: TF32 products would not hold the 1e-5 fp32 bound.  Every
// kernel is instantiated for d = 64 and d = 128 (template parameter D).
#include "da_internal.h"

#include <cuda_bf16.h>

namespace da {

constexpr int kF32RowsPerCta = 64;
constexpr int kF32KeysPerCta = 128;
constexpr int kF32QChunk = 32;

template <int D>
__global__ void __launch_bounds__(kF32RowsPerCta)
    f32_rowstats(const float *__restrict__ q, const float *__restrict__ k, float *__restrict__ lse2,
                 float *__restrict__ acc, int T, int Tp, HeadScale hs, int *status) {
  constexpr int AS = acc_stride(D);
  __shared__ float sk[kF32RowsPerCta][D];
  const int bh = blockIdx.y;
  const float c2 = head_c2(hs, bh, threadIdx.x == 0 ? status : nullptr);
  const int tid = threadIdx.x;
  const int i = blockIdx.x * kF32RowsPerCta + tid;
  const float *qb = q + (size_t)bh * T * D;
  const float *kb = k + (size_t)bh * T * D;

  float qr[D];
#pragma unroll
  for (int t = 0; t < D; ++t) qr[t] = (i < T) ? qb[(size_t)i * D + t] : 0.f;

  float m = -INFINITY, l = 0.f;
  const int last_key = min(blockIdx.x * kF32RowsPerCta + kF32RowsPerCta - 1, T - 1);
  for (int k0 = 0; k0 <= last_key; k0 += kF32RowsPerCta) {
    __syncthreads();
    const int kr = k0 + tid;
#pragma unroll 4
    for (int t = 0; t < D; ++t) sk[tid][t] = (kr < T) ? kb[(size_t)kr * D + t] : 0.f;
    __syncthreads();
    for (int kk = 0; kk < kF32RowsPerCta; ++kk) {
      const int key = k0 + kk;
      if (!visible(i, key, T)) continue;
      float s = 0.f;
#pragma unroll
      for (int t = 0; t < D; ++t) s = fmaf(qr[t], sk[kk][t], s);
      // max in fl(s*c2); every term of the sum as fma(s, c2, -m), so no
      // term carries the rounding of a large logit.
      const float x = s * c2;
      if (x > m) {
        l = l * exp2f(m - x) + exp2f(fmaf(s, c2, -x));
        m = x;
      } else {
        l += exp2f(fmaf(s, c2, -m));
      }
    }
  }
  if (i < Tp) {
    // The normaliser is kept as (m, log2 l): at logits of magnitude ~30 a
    // single fp32 lse2 would carry ~2e-6 absolute rounding into every bid.
    // m goes to the lse2 slot, log2 l to pad column d + 1 of the accumulator row.
    lse2[(size_t)bh * Tp + i] = (i < T) ? m : INFINITY;
    float4 *ar = reinterpret_cast<float4 *>(acc + ((size_t)bh * Tp + i) * AS);
#pragma unroll
    for (int t = 0; t < AS / 4; ++t) ar[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[((size_t)bh * Tp + i) * AS + D + 1] = (i < T) ? log2f(l) : 0.f;
  }
}

template <int D>
struct F32SweepSmem {
  float v[kF32KeysPerCta][D];                  // value rows of this CTA's keys
  float q[kF32QChunk][D];                      // current query chunk
  float m2[kF32QChunk];                        // its row maxima (log2 domain)
  float ll[kF32QChunk];                        // and log2 of the normalisers
  float sh[kF32QChunk][kF32KeysPerCta + 1];    // shares [query][key]
};

template <int D>
__global__ void __launch_bounds__(kF32KeysPerCta)
    f32_sweep(const float *__restrict__ q, const float *__restrict__ k, const float *__restrict__ v,
              const float *__restrict__ lse2, float *__restrict__ acc, float *__restrict__ demand_out, int T,
              int Tp, HeadScale hs, float eps, bool earlier) {
  extern __shared__ float4 f32_smem_raw[];
  constexpr int AS = acc_stride(D);
  F32SweepSmem<D> &S = *reinterpret_cast<F32SweepSmem<D> *>(f32_smem_raw);
  const int bh = blockIdx.y;
  const float c2 = head_c2(hs, bh, nullptr);   // the row statistics report bad entries
  const int tid = threadIdx.x;
  const int key0 = blockIdx.x * kF32KeysPerCta;
  const int key = key0 + tid;
  const float *qb = q + (size_t)bh * T * D;
  const float *kb = k + (size_t)bh * T * D;
  const float *vb = v + (size_t)bh * T * D;

  float kr[D];
#pragma unroll
  for (int t = 0; t < D; ++t) kr[t] = (key < T) ? kb[(size_t)key * D + t] : 0.f;
#pragma unroll 4
  for (int t = 0; t < D; ++t) S.v[tid][t] = (key < T) ? vb[(size_t)key * D + t] : 0.f;

  float committed = 0.f;   // sum of bids this key received from earlier queries
  float comp = 0.f;        // Kahan compensation of that sum
  constexpr int RG = kF32KeysPerCta / D;       // row groups of the numerator step
  const int dv = tid % D;
  const int rhalf = tid / D;
  for (int q0 = key0; q0 < T; q0 += kF32QChunk) {
    __syncthreads();
    for (int e = tid; e < kF32QChunk * D; e += kF32KeysPerCta) {
      const int r = e / D, t = e % D;
      S.q[r][t] = (q0 + r < T) ? qb[(size_t)(q0 + r) * D + t] : 0.f;
    }
    if (tid < kF32QChunk) {
      S.m2[tid] = lse2[(size_t)bh * Tp + q0 + tid];
      S.ll[tid] = acc[((size_t)bh * Tp + q0 + tid) * AS + D + 1];
    }
    __syncthreads();
    for (int r = 0; r < kF32QChunk; ++r) {
      const int i = q0 + r;
      float share = 0.f;
      if (visible(i, key, T)) {
        float s = 0.f;
#pragma unroll
        for (int t = 0; t < D; ++t) s = fmaf(S.q[r][t], kr[t], s);
        const float p = exp2f(fmaf(s, c2, -S.m2[r]) - S.ll[r]);
        share = p / ((earlier ? committed : committed + p) + eps);
        const float y = p - comp;
        const float t2 = committed + y;
        comp = (t2 - committed) - y;
        committed = t2;
      }
      S.sh[r][tid] = share;
    }
    __syncthreads();
    // Partial numerators: thread (rhalf, dv) owns 32 / RG query rows of column dv.
    for (int rr = 0; rr < kF32QChunk / RG; ++rr) {
      const int r = rhalf * (kF32QChunk / RG) + rr;
      if (q0 + r >= T) break;
      float a = 0.f;
      for (int kk = 0; kk < kF32KeysPerCta; ++kk) a = fmaf(S.sh[r][kk], S.v[kk][dv], a);
      atomicAdd(acc + ((size_t)bh * Tp + q0 + r) * AS + dv, a);
    }
    if (tid < kF32QChunk && q0 + tid < T) {
      float rs = 0.f;
      for (int kk = 0; kk < kF32KeysPerCta; ++kk) rs += S.sh[tid][kk];
      atomicAdd(acc + ((size_t)bh * Tp + q0 + tid) * AS + D, rs);
    }
  }
  if (demand_out != nullptr && key < T) demand_out[(size_t)bh * T + key] = committed;
}

// out_i = acc_i[0:d] / acc_i[d]; optional rowsum and lse2 side outputs.
// d / 4 threads per row, 4 columns each.
// split_lse: the workspace holds the row max and log2(l) separately (fp32
// path); otherwise it holds -lse2 (bf16 path).
constexpr int kFinRows = 4;

template <typename OutT, int D>
__global__ void finalize_kernel(const float *__restrict__ acc, const float *__restrict__ lse2_ws,
                                OutT *__restrict__ out, float *__restrict__ rowsum_out,
                                float *__restrict__ lse2_out, int BH, int T, int Tp, bool split_lse) {
  // TPR threads per row (one float4 of the numerator each); every thread
  // handles kFinRows rows spaced one grid apart, with all loads issued before
  // any arithmetic so that enough bytes are in flight for HBM rate.
  constexpr int TPR = D / 4, AS = acc_stride(D);
  const int64_t nrows = (int64_t)BH * T;
  const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x / TPR;   // rows per grid
  const int part = (int)(g % TPR);
  float rs[kFinRows];
  float4 a[kFinRows];
#pragma unroll
  for (int j = 0; j < kFinRows; ++j) {
    const int64_t row = g / TPR + j * stride;
    if (row < nrows) {
      const int64_t bh = row / T, i = row % T;
      const float *ar = acc + ((size_t)bh * Tp + i) * AS;
      rs[j] = __ldg(ar + D);
      a[j] = __ldg(reinterpret_cast<const float4 *>(ar) + part);
    }
  }
#pragma unroll
  for (int j = 0; j < kFinRows; ++j) {
    const int64_t row = g / TPR + j * stride;
    if (row >= nrows) break;
    const float inv = 1.f / rs[j];
    if constexpr (sizeof(OutT) == 4) {
      reinterpret_cast<float4 *>(out + row * D)[part] =
          make_float4(a[j].x * inv, a[j].y * inv, a[j].z * inv, a[j].w * inv);
    } else {
      __nv_bfloat162 lo = __floats2bfloat162_rn(a[j].x * inv, a[j].y * inv);
      __nv_bfloat162 hi = __floats2bfloat162_rn(a[j].z * inv, a[j].w * inv);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t *>(&lo);
      pk.y = *reinterpret_cast<uint32_t *>(&hi);
      reinterpret_cast<uint2 *>(out + row * D)[part] = pk;
    }
    if (part == 0) {
      const int64_t bh = row / T, i = row % T;
      if (rowsum_out) rowsum_out[row] = rs[j];
      if (lse2_out)
        lse2_out[row] = split_lse ? lse2_ws[(size_t)bh * Tp + i] + acc[((size_t)bh * Tp + i) * AS + D + 1]
                                  : -lse2_ws[(size_t)bh * Tp + i];
    }
  }
}

// Grid of the finalize pass: d / 4 threads per row, kFinRows rows per thread.
static unsigned finalize_blocks(int64_t nrows, int d) {
  const int64_t threads = (nrows + kFinRows - 1) / kFinRows * (d / 4);
  return (unsigned)((threads + 255) / 256);
}

// ------------------------------------------------------------ host launchers
template <int D>
static cudaError_t launch_fwd_f32_t(const float *q, const float *k, const float *v, float *out, float *lse2_out,
                                    float *rowsum_out, float *demand_out, int BH, int T, HeadScale hs, float eps,
                                    bool earlier, float *lse2_ws, float *acc, int *status, cudaStream_t stream,
                                    cudaEvent_t const *ev) {
  const int Tp = (int)t_pad(T);
  if (ev[0]) cudaEventRecord(ev[0], stream);
  f32_rowstats<D><<<dim3(Tp / kF32RowsPerCta, BH), kF32RowsPerCta, 0, stream>>>(q, k, lse2_ws, acc, T, Tp, hs,
                                                                                 status);
  const size_t smem = sizeof(F32SweepSmem<D>);
  cudaError_t e = cudaFuncSetAttribute(f32_sweep<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  if (ev[1]) cudaEventRecord(ev[1], stream);
  f32_sweep<D><<<dim3(Tp / kF32KeysPerCta, BH), kF32KeysPerCta, smem, stream>>>(q, k, v, lse2_ws, acc, demand_out,
                                                                               T, Tp, hs, eps, earlier);
  if (ev[2]) cudaEventRecord(ev[2], stream);
  finalize_kernel<float, D><<<finalize_blocks((int64_t)BH * T, D), 256, 0, stream>>>(acc, lse2_ws, out, rowsum_out,
                                                                                    lse2_out, BH, T, Tp, true);
  if (ev[3]) cudaEventRecord(ev[3], stream);
  return cudaGetLastError();
}

cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *out, float *lse2_out,
                           float *rowsum_out, float *demand_out, int BH, int T, int d, HeadScale hs, float eps,
                           bool earlier, float *lse2_ws, float *acc, int *status, cudaStream_t stream,
                           cudaEvent_t const *ev) {
  if (d == 128)
    return launch_fwd_f32_t<128>(q, k, v, out, lse2_out, rowsum_out, demand_out, BH, T, hs, eps, earlier, lse2_ws,
                                 acc, status, stream, ev);
  return launch_fwd_f32_t<64>(q, k, v, out, lse2_out, rowsum_out, demand_out, BH, T, hs, eps, earlier, lse2_ws, acc,
                              status, stream, ev);
}

cudaError_t launch_finalize_bf16(const float *acc, const float *lse2_ws, __nv_bfloat16 *out, float *rowsum_out,
                                 float *lse2_out, int BH, int T, int d, cudaStream_t stream) {
  const int Tp = (int)t_pad(T);
  if (d == 128)
    finalize_kernel<__nv_bfloat16, 128><<<finalize_blocks((int64_t)BH * T, 128), 256, 0, stream>>>(
        acc, lse2_ws, out, rowsum_out, lse2_out, BH, T, Tp, false);
  else
    finalize_kernel<__nv_bfloat16, 64><<<finalize_blocks((int64_t)BH * T, 64), 256, 0, stream>>>(
        acc, lse2_ws, out, rowsum_out, lse2_out, BH, T, Tp, false);
  return cudaGetLastError();
}

}  // namespace da
