// C ABI of the dilution-attention library: argument validation, workspace
// layout, dispatch to the kernels, status reporting and host-only debug
// exports of the integer artefacts (tile schedules, causal mask).
#include <cmath>
#include <cstring>

#include <cuda_bf16.h>

#include "da_internal.h"

namespace da {
cudaError_t launch_fwd_f32(const float *q, const float *k, const float *v, float *out, float *lse2_out,
                           float *rowsum_out, float *demand_out, int BH, int T, int d, HeadScale hs, float eps,
                           bool earlier, float *lse2_ws, float *acc, int *status, cudaStream_t stream,
                           cudaEvent_t const *ev);
int launch_fwd_bf16(const void *q, const void *k, const void *v, void *out, float *lse2_out, float *rowsum_out,
                    float *demand_out, int BH, int T, int d, HeadScale hs, float eps, bool earlier, float *lse2_ws,
                    float *acc, float *cchk, int *status, cudaStream_t stream, cudaEvent_t const *ev);
cudaError_t launch_bwd(const void *q, const void *k, const void *v, const void *dout, const float *lse2, void *dq,
                       void *dk, void *dv, int BH, int T, int d, float c, HeadScale hs, float eps, bool earlier,
                       int dtype, double *dtot, float *rowbuf, float *dq_acc, cudaStream_t stream);
int launch_bwd_bf16_tc(const void *q, const void *k, const void *v, const void *dout, const float *lse2, void *dq,
                       void *dk, void *dv, int BH, int T, int d, HeadScale hs, float c, float eps, bool earlier,
                       bool have_fwd_state, uint8_t *ws, cudaStream_t stream);
cudaError_t launch_decode(const void *q_new, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          float *demand, int n_ctx, int T_cap, void *out, int BH, int d, HeadScale hs, float eps,
                          bool earlier, int dtype, float *logits, float2 *part_ml, float *part_acc, int nchunk,
                          int *status, DecDebug dbg, cudaStream_t stream);
}  // namespace da

using namespace da;

namespace {

constexpr double kLog2e = 1.4426950408889634;
// The kernels' bounded-wait limit (1 s), as the host sees it.
constexpr unsigned long long kWaitLimitNsHost = 1000ull * 1000ull * 1000ull;

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned16_or_null(const void *p) { return p == nullptr || aligned16(p); }

// Scale applied to q.k in the log2 domain: tau / sqrt(d) * log2(e).
double log2e_over_sqrt_d(int d) { return kLog2e / std::sqrt((double)d); }
float logit_scale_log2(float tau, int d) { return (float)((double)tau * log2e_over_sqrt_d(d)); }

HeadScale head_scale(float tau, const float *tau_bh, int d) {
  return HeadScale{tau_bh, logit_scale_log2(tau, d), log2e_over_sqrt_d(d)};
}

// bf16 runs the tensor-core backward; fp32 the SIMT one.
bool bwd_on_tensor_cores(int d, int dtype) { return dtype == DA_BF16 && (d == 64 || d == 128); }

// Options of the *_ex entry points.
int check_options(const float *tau_bh, int flags) {
  if ((flags & ~(DA_FLAG_EARLIER_DEMAND_ONLY | DA_FLAG_KEEP_FOR_BACKWARD)) != 0) return DA_ERR_INVALID;
  if ((reinterpret_cast<uintptr_t>(tau_bh) & 3u) != 0) return DA_ERR_INVALID;
  return DA_OK;
}

int check_common(int B, int H, int T, int d, float tau, float eps, int dtype) {
  if (B < 0 || H < 0 || T < 0) return DA_ERR_INVALID;
  if (!std::isfinite(tau) || tau < 0.f) return DA_ERR_INVALID;
  if (!std::isfinite(eps) || eps <= 0.f) return DA_ERR_INVALID;
  if (dtype != DA_F32 && dtype != DA_BF16) return DA_ERR_INVALID;
  if (!head_dim_supported(d)) return DA_ERR_UNSUPPORTED;
  if (T > DA_MAX_T) return DA_ERR_UNSUPPORTED;
  if ((int64_t)B * H > (1 << 24)) return DA_ERR_UNSUPPORTED;
  return DA_OK;
}

}  // namespace

extern "C" {

const char *dilution_attn_status_string(int status) {
  switch (status) {
    case DA_OK: return "DA_OK";
    case DA_ERR_INVALID: return "DA_ERR_INVALID: invalid argument";
    case DA_ERR_UNSUPPORTED: return "DA_ERR_UNSUPPORTED: unsupported shape or dtype";
    case DA_ERR_CUDA: return "DA_ERR_CUDA: CUDA runtime call failed";
    case DA_ERR_TIMEOUT: return "DA_ERR_TIMEOUT: a kernel wait timed out";
    case DA_ERR_WORKSPACE: return "DA_ERR_WORKSPACE: workspace missing or too small";
    default: return "unknown status";
  }
}

int dilution_attn_version(void) { return 101; }

size_t dilution_attn_fwd_workspace_size(int B, int H, int T, int d, int dtype) {
  (void)dtype;
  if (B < 0 || H < 0 || T < 0 || !head_dim_supported(d)) return 0;
  return fwd_workspace_layout((int64_t)B * H, T, d).total;
}

int dilution_attn_fwd(const void *q, const void *k, const void *v, void *out, float *lse2_out, float *rowsum_out,
                      float *demand_out, int B, int H, int T, int d, float tau, float eps, int dtype,
                      void *workspace, size_t workspace_bytes, void *stream_) {
  return dilution_attn_fwd_ex(q, k, v, out, lse2_out, rowsum_out, demand_out, B, H, T, d, tau, nullptr, eps, 0,
                              dtype, workspace, workspace_bytes, stream_, nullptr);
}

int dilution_attn_fwd_with_events(const void *q, const void *k, const void *v, void *out, float *lse2_out,
                                  float *rowsum_out, float *demand_out, int B, int H, int T, int d, float tau,
                                  float eps, int dtype, void *workspace, size_t workspace_bytes, void *stream_,
                                  void *const *events) {
  return dilution_attn_fwd_ex(q, k, v, out, lse2_out, rowsum_out, demand_out, B, H, T, d, tau, nullptr, eps, 0,
                              dtype, workspace, workspace_bytes, stream_, events);
}

int dilution_attn_fwd_ex(const void *q, const void *k, const void *v, void *out, float *lse2_out,
                         float *rowsum_out, float *demand_out, int B, int H, int T, int d, float tau,
                         const float *tau_bh, float eps, int flags, int dtype, void *workspace,
                         size_t workspace_bytes, void *stream_, void *const *events) {
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
  if (events != nullptr)
    for (int i = 0; i < 4; ++i) ev[i] = reinterpret_cast<cudaEvent_t>(events[i]);
  int st = check_common(B, H, T, d, tau, eps, dtype);
  if (st == DA_OK) st = check_options(tau_bh, flags);
  if (st != DA_OK) return st;
  const bool earlier = (flags & DA_FLAG_EARLIER_DEMAND_ONLY) != 0;
  const int64_t BH = (int64_t)B * H;
  if (BH == 0 || T == 0) return DA_OK;
  if (q == nullptr || k == nullptr || v == nullptr || out == nullptr) return DA_ERR_INVALID;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return DA_ERR_INVALID;
  if (!aligned16_or_null(lse2_out) || !aligned16_or_null(rowsum_out) || !aligned16_or_null(demand_out))
    return DA_ERR_INVALID;
  // DA_FLAG_KEEP_FOR_BACKWARD: the workspace is a backward workspace whose
  // leading regions (-lse2, accumulators) are laid out as the forward's; the
  // sweep also writes the demand checkpoints there.
  const bool keep = (flags & DA_FLAG_KEEP_FOR_BACKWARD) != 0;
  if (keep && !bwd_on_tensor_cores(d, dtype)) return DA_ERR_UNSUPPORTED;
  const FwdWorkspace L = fwd_workspace_layout(BH, T, d);
  const BwdTcWorkspace LB = bwd_tc_workspace_layout(BH, T, d);
  if (keep && (LB.nlse2_off != L.lse2_off || LB.acc_off != L.acc_off)) return DA_ERR_UNSUPPORTED;
  if (workspace == nullptr || workspace_bytes < (keep ? LB.total : L.total)) return DA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DA_ERR_INVALID;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
  int *status = reinterpret_cast<int *>(ws);
  float *lse2_ws = reinterpret_cast<float *>(ws + L.lse2_off);
  float *acc = reinterpret_cast<float *>(ws + L.acc_off);
  float *cchk = keep ? reinterpret_cast<float *>(ws + LB.cchk_off) : nullptr;
  if (dtype == DA_BF16 && eps < 1e-18f) return DA_ERR_UNSUPPORTED;
  if (cudaMemsetAsync(status, 0, kStatusWordsReset * sizeof(int), stream) != cudaSuccess) return DA_ERR_CUDA;
  const HeadScale hs = head_scale(tau, tau_bh, d);
  if (dtype == DA_F32) {
    if (launch_fwd_f32((const float *)q, (const float *)k, (const float *)v, (float *)out, lse2_out, rowsum_out,
                       demand_out, (int)BH, T, d, hs, eps, earlier, lse2_ws, acc, status, stream, ev) != cudaSuccess)
      return DA_ERR_CUDA;
    return DA_OK;
  }
  return launch_fwd_bf16(q, k, v, out, lse2_out, rowsum_out, demand_out, (int)BH, T, d, hs, eps, earlier, lse2_ws,
                         acc, cchk, status, stream, ev);
}

size_t dilution_attn_bwd_workspace_size(int B, int H, int T, int d, int dtype) {
  if (B < 0 || H < 0 || T < 0 || !head_dim_supported(d)) return 0;
  if (bwd_on_tensor_cores(d, dtype)) return bwd_tc_workspace_layout((int64_t)B * H, T, d).total;
  return bwd_workspace_layout((int64_t)B * H, T, d).total;
}

int dilution_attn_bwd(const void *q, const void *k, const void *v, const void *dout, const float *lse2, void *dq,
                      void *dk, void *dv, int B, int H, int T, int d, float tau, float eps, int dtype,
                      void *workspace, size_t workspace_bytes, void *stream_) {
  return dilution_attn_bwd_ex(q, k, v, dout, lse2, dq, dk, dv, B, H, T, d, tau, nullptr, eps, 0, dtype, workspace,
                              workspace_bytes, stream_);
}

int dilution_attn_bwd_ex(const void *q, const void *k, const void *v, const void *dout, const float *lse2,
                         void *dq, void *dk, void *dv, int B, int H, int T, int d, float tau, const float *tau_bh,
                         float eps, int flags, int dtype, void *workspace, size_t workspace_bytes, void *stream_) {
  int st = check_common(B, H, T, d, tau, eps, dtype);
  if (st == DA_OK) st = check_options(tau_bh, flags);
  if (st != DA_OK) return st;
  const bool keep = (flags & DA_FLAG_KEEP_FOR_BACKWARD) != 0;
  if (keep && !bwd_on_tensor_cores(d, dtype)) return DA_ERR_UNSUPPORTED;
  const int64_t BH = (int64_t)B * H;
  if (BH == 0 || T == 0) return DA_OK;
  const void *ptrs[] = {q, k, v, dout, lse2, dq, dk, dv};
  for (const void *p : ptrs)
    if (p == nullptr || !aligned16(p)) return DA_ERR_INVALID;
  const size_t need = bwd_on_tensor_cores(d, dtype) ? bwd_tc_workspace_layout(BH, T, d).total
                                                   : bwd_workspace_layout(BH, T, d).total;
  if (workspace == nullptr || workspace_bytes < need) return DA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DA_ERR_INVALID;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
  if (cudaMemsetAsync(ws, 0, 4 * sizeof(int), stream) != cudaSuccess) return DA_ERR_CUDA;
  const float c = (float)((double)tau / std::sqrt((double)d));
  if (bwd_on_tensor_cores(d, dtype)) {
    if ((int64_t)BH * t_pad(T) > 0x7FFFFFFF) return DA_ERR_UNSUPPORTED;
    return launch_bwd_bf16_tc(q, k, v, dout, lse2, dq, dk, dv, (int)BH, T, d, head_scale(tau, tau_bh, d), c, eps,
                              (flags & DA_FLAG_EARLIER_DEMAND_ONLY) != 0, keep, ws, stream);
  }
  const BwdWorkspace L = bwd_workspace_layout(BH, T, d);
  if (launch_bwd(q, k, v, dout, lse2, dq, dk, dv, (int)BH, T, d, c, head_scale(tau, tau_bh, d), eps,
                 (flags & DA_FLAG_EARLIER_DEMAND_ONLY) != 0, dtype,
                 reinterpret_cast<double *>(ws + L.dtot_off), reinterpret_cast<float *>(ws + L.row_off),
                 reinterpret_cast<float *>(ws + L.dq_off), stream) != cudaSuccess)
    return DA_ERR_CUDA;
  return DA_OK;
}

size_t dilution_attn_decode_workspace_size(int B, int H, int T_cap, int d) {
  if (B < 0 || H < 0 || T_cap < 0 || !head_dim_supported(d)) return 0;
  return dec_workspace_layout((int64_t)B * H, T_cap, d).total;
}

int dilution_attn_decode_step(const void *q_new, const void *k_new, const void *v_new, void *k_cache,
                              void *v_cache, float *demand, int n_ctx, int T_cap, void *out, int B, int H, int d,
                              float tau, float eps, int dtype, void *workspace, size_t workspace_bytes,
                              void *stream_) {
  return dilution_attn_decode_step_ex(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx, T_cap, out, B, H, d, tau,
                                      nullptr, eps, 0, dtype, workspace, workspace_bytes, stream_);
}

}  // extern "C"

namespace da {
// Argument checks of a decode step that need no workspace: sizes, tau, eps,
// dtype, options, n_ctx and the tensor pointers.  Returns DA_OK, or the status
// the step returns for them (B * H == 0 passes: the step then does nothing).
int check_decode_step_args(const void *q_new, const void *k_new, const void *v_new, const void *k_cache,
                           const void *v_cache, const float *demand, int n_ctx, int T_cap, const void *out, int B,
                           int H, int d, float tau, const float *tau_bh, float eps, int flags, int dtype) {
  int st = check_common(B, H, T_cap, d, tau, eps, dtype);
  if (st == DA_OK) st = check_options(tau_bh, flags);
  if (st != DA_OK) return st;
  if ((flags & DA_FLAG_KEEP_FOR_BACKWARD) != 0) return DA_ERR_INVALID;   // no backward of a decode step
  if (n_ctx < 0 || n_ctx >= T_cap) return DA_ERR_INVALID;
  if ((int64_t)B * H == 0) return DA_OK;
  const void *ptrs[] = {q_new, k_new, v_new, k_cache, v_cache, demand, out};
  for (const void *p : ptrs)
    if (p == nullptr || !aligned16(p)) return DA_ERR_INVALID;
  return DA_OK;
}
}  // namespace da

namespace {
// The decode step behind dilution_attn_decode_step_ex and its test hook.
int decode_step_impl(const void *q_new, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                     float *demand, int n_ctx, int T_cap, void *out, int B, int H, int d, float tau,
                     const float *tau_bh, float eps, int flags, int dtype, void *workspace, size_t workspace_bytes,
                     void *stream_, DecDebug dbg) {
  const int st = check_decode_step_args(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx, T_cap, out, B, H, d,
                                        tau, tau_bh, eps, flags, dtype);
  if (st != DA_OK) return st;
  const int64_t BH = (int64_t)B * H;
  if (BH == 0) return DA_OK;
  const DecWorkspace L = dec_workspace_layout(BH, T_cap, d);
  if (workspace == nullptr || workspace_bytes < L.total) return DA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return DA_ERR_INVALID;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  uint8_t *ws = reinterpret_cast<uint8_t *>(workspace);
  if (cudaMemsetAsync(ws, 0, 4 * sizeof(int), stream) != cudaSuccess) return DA_ERR_CUDA;
  if (launch_decode(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx, T_cap, out, (int)BH, d,
                    head_scale(tau, tau_bh, d), eps, (flags & DA_FLAG_EARLIER_DEMAND_ONLY) != 0, dtype,
                    reinterpret_cast<float *>(ws + L.logit_off), reinterpret_cast<float2 *>(ws + L.ml_off),
                    reinterpret_cast<float *>(ws + L.acc_off), L.nchunk, reinterpret_cast<int *>(ws), dbg,
                    stream) != cudaSuccess)
    return DA_ERR_CUDA;
  return DA_OK;
}
}  // namespace

extern "C" {

int dilution_attn_decode_step_ex(const void *q_new, const void *k_new, const void *v_new, void *k_cache,
                                 void *v_cache, float *demand, int n_ctx, int T_cap, void *out, int B, int H, int d,
                                 float tau, const float *tau_bh, float eps, int flags, int dtype, void *workspace,
                                 size_t workspace_bytes, void *stream_) {
  return decode_step_impl(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx, T_cap, out, B, H, d, tau, tau_bh, eps,
                          flags, dtype, workspace, workspace_bytes, stream_, DecDebug{kWaitLimitNsHost, -1, -1});
}

int dilution_attn_debug_decode_stall(const void *q_new, const void *k_new, const void *v_new, void *k_cache,
                                     void *v_cache, float *demand, int n_ctx, int T_cap, void *out, int B, int H,
                                     int d, float tau, float eps, int dtype, void *workspace, size_t workspace_bytes,
                                     void *stream_, int stall_chunk, int stall_bh, long long wait_limit_ns) {
  if (wait_limit_ns < 1000 || wait_limit_ns > (long long)kWaitLimitNsHost) return DA_ERR_INVALID;
  if (stall_chunk < 0 || stall_bh < 0 || (int64_t)stall_bh >= (int64_t)B * H) return DA_ERR_INVALID;
  return decode_step_impl(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx, T_cap, out, B, H, d, tau, nullptr,
                          eps, 0, dtype, workspace, workspace_bytes, stream_,
                          DecDebug{(unsigned long long)wait_limit_ns, stall_chunk, stall_bh});
}

int dilution_attn_get_error(void *workspace, void *stream_) {
  if (workspace == nullptr) return DA_ERR_INVALID;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int host = 0;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DA_ERR_CUDA;
  if (cudaMemcpy(&host, workspace, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DA_ERR_CUDA;
  if (host != DA_OK && cudaMemset(workspace, 0, sizeof(int)) != cudaSuccess) return DA_ERR_CUDA;
  return host;
}

int dilution_attn_debug_last_timeout(void *workspace, int32_t *out) {
  if (workspace == nullptr || out == nullptr) return DA_ERR_INVALID;
  if (cudaDeviceSynchronize() != cudaSuccess) return DA_ERR_CUDA;
  if (cudaMemcpy(out, workspace, 4 * sizeof(int32_t), cudaMemcpyDeviceToHost) != cudaSuccess) return DA_ERR_CUDA;
  return DA_OK;
}

int dilution_attn_debug_tile_schedule(int BH, int T, int kernel, int32_t *out, size_t cap) {
  if (BH < 0 || T < 0 || kernel < 0 || kernel > 9) return -1;
  if (BH == 0 || T == 0) return 0;
  // kernel 0: row statistics at d = 64, 1: sweep at d = 64, 2: sweep at
  // d = 128, 3: row statistics at d = 128; 4 + 2 pass + (d == 128): the
  // backward's reverse pass (pass 0), light dK pass (1) and dQ pass (2)
  const bool rs = kernel == 0 || kernel == 3, bwd = kernel >= 4;
  const int d = bwd ? ((kernel - 4) % 2 ? 128 : 64) : (kernel == 2 || kernel == 3 ? 128 : 64);
  const int pass = bwd ? (kernel - 4) / 2 : 0;
  const int n = bwd ? bwd_num_ctas(BH, T) : rs ? rowstats_num_ctas(BH, T) : sweep_num_ctas(BH, T, d);
  if (out == nullptr || cap < (size_t)n * 4) return -n;
  for (int c = 0; c < n; ++c) {
    const TileWork w = bwd  ? bwd_work(c, BH, T, d, pass)
                       : rs ? rowstats_work(c, BH, T, d)
                            : sweep_work(c, BH, T, d);
    out[4 * c + 0] = w.bh;
    out[4 * c + 1] = w.q_tile0;
    out[4 * c + 2] = w.n_q_tiles;
    out[4 * c + 3] = w.key0;
  }
  return n;
}

int dilution_attn_debug_tile_mask(int T, int qt, int kt, uint8_t *out) {
  if (T < 0 || qt < 0 || kt < 0 || out == nullptr) return DA_ERR_INVALID;
  for (int r = 0; r < kTile; ++r)
    for (int c = 0; c < kTile; ++c)
      out[r * kTile + c] = visible((int64_t)qt * kTile + r, (int64_t)kt * kTile + c, T) ? 1 : 0;
  return DA_OK;
}

}  // extern "C"
