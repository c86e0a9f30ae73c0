/*
 * dilution_attn.h -- C ABI of the GB300 (sm_103a) dilution-attention library.
 *
 * The operator ("DilutionAttention v0.1.0 · results", section "The operator"):
 * for every (batch b, head h) independently, with queries i and keys k,
 *
 *     s_ik      = tau * (q_i . k_k) / sqrt(d)                    (k <= i only)
 *     p_ik      = exp(s_ik) / sum_{k' <= i} exp(s_ik')           causal softmax: the bids
 *     committed = sum_{j < i} p_jk                               demand from earlier queries
 *     share_ik  = p_ik / (committed_ik + p_ik + eps)
 *     out_i     = sum_k share_ik v_k / sum_k share_ik             A = share / rowsum(share)
 *
 * tau is a logit multiplier (1 by default).  A focal temperature t
 * ("Focal Attention", arXiv 2511.06818, section "Transformer with Constant
 * Temperature", eq. focal-const) is tau = 1/t; YaRN's sharpening
 * ("YaRN › Attention Temperature Scaling", temperature formula) is
 * tau = sqrt(0.1 ln s + 1).
 *
 * Conventions shared by every entry point
 *   - Layout: q, k, v, out are contiguous [B, H, T, d] (d fastest); per-row
 *     vectors (lse2, rowsum, demand) are contiguous [B, H, T].
 *   - Pointers are DEVICE pointers unless stated otherwise, 16-byte aligned.
 *     The caller owns every buffer; the library allocates nothing and keeps
 *     no state between calls.  Scratch memory is the caller's workspace.
 *   - stream is a cudaStream_t (NULL = legacy default stream).  Compute
 *     calls are asynchronous: argument errors are returned synchronously
 *     before anything is enqueued; kernel-side errors (a bounded wait that
 *     timed out) are written to a status word at the start of the workspace
 *     and read back with dilution_attn_get_error().
 *   - Supported: d == 64 or d == 128 (other head sizes return
 *     DA_ERR_UNSUPPORTED and a workspace size of 0); dtype DA_F32 (fp32
 *     in/out, fp32 SIMT arithmetic) or DA_BF16 (bf16 in/out, bf16
 *     tensor-core products, fp32 accumulation and fp32 softmax/demand
 *     arithmetic).  tau >= 0 and finite; eps > 0 and
 *     finite (eps = 0 would make masked and underflowed entries 0/0).
 *     B, H, T >= 0; a call with B*H*T == 0 does nothing and returns DA_OK.
 *     T <= DA_MAX_T.  The DA_BF16 forward needs eps >= 1e-18 (it forms one
 *     reciprocal for each pair of denominators, each >= eps); smaller eps
 *     returns DA_ERR_UNSUPPORTED.
 */
#ifndef DILUTION_ATTN_H
#define DILUTION_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every call. */
#define DA_OK              0
#define DA_ERR_INVALID     1   /* bad argument: null/misaligned pointer, negative size, eps <= 0, ... */
#define DA_ERR_UNSUPPORTED 2   /* valid but not implemented: d not 64 or 128, T > DA_MAX_T, ...   */
#define DA_ERR_CUDA        3   /* a CUDA runtime call failed (launch, tensor-map encode, copy)   */
#define DA_ERR_TIMEOUT     4   /* a kernel's bounded wait expired; results are not valid         */
#define DA_ERR_WORKSPACE   5   /* workspace pointer null or smaller than the *_workspace_size    */

/* Element types. */
#define DA_F32  0
#define DA_BF16 1

#define DA_MAX_T (1 << 24)

/* Flags of the *_ex entry points (bitwise or; other bits are DA_ERR_INVALID). */
#define DA_FLAG_EARLIER_DEMAND_ONLY 1   /* share = p / (committed + eps): see below */
#define DA_FLAG_KEEP_FOR_BACKWARD   2   /* forward leaves its state for the backward: see below */

/* Human-readable name of a status code (static string, never NULL). */
const char *dilution_attn_status_string(int status);

/* Library ABI version (major*100 + minor). */
int dilution_attn_version(void);

/* ------------------------------------------------------------------------
 * Prefill forward.
 *
 * Computes out for all T queries of each (b, h) (the operator above), plus
 * optional per-row side outputs:
 *   lse2_out   [B,H,T] fp32, nullable: log2 of the softmax normaliser of the
 *              scaled logits, log2(sum_{k<=i} 2^(s_ik * log2 e)); the bid is
 *              p_ik = 2^(s_ik*log2 e - lse2_i).
 *   rowsum_out [B,H,T] fp32, nullable: R_i = sum_k share_ik, the normaliser
 *              of row i of A = share / R (whose rows therefore sum to 1 by
 *              construction); out_i = sum_k share_ik v_k / R_i.
 *   demand_out [B,H,T] fp32, nullable: column totals sum_i p_ik over all T
 *              queries -- the decode demand cache after prefill
 *              ("DilutionAttention v0.1.0 · results", section "The operator",
 *              cached decoding).
 * workspace: device scratch of at least dilution_attn_fwd_workspace_size()
 * bytes; its first 256 bytes hold the status word.  For bf16 inputs, int32
 * word 4 of that block counts the rows whose softmax normaliser the
 * tensor-core pass handed to an exact per-row recomputation (its running sum
 * overflowed: a logit more than ~106 log2 units above the maximum of the
 * row's first 32 keys); diagnostic only.  Every call overwrites the
 * workspace, so concurrent calls on different streams need distinct
 * workspaces.  Errors: DA_ERR_INVALID, DA_ERR_UNSUPPORTED, DA_ERR_WORKSPACE,
 * DA_ERR_CUDA (launch failure).
 * ---------------------------------------------------------------------- */
size_t dilution_attn_fwd_workspace_size(int B, int H, int T, int d, int dtype);

int dilution_attn_fwd(const void *q, const void *k, const void *v, void *out,
                      float *lse2_out, float *rowsum_out, float *demand_out,
                      int B, int H, int T, int d, float tau, float eps, int dtype,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Same computation as dilution_attn_fwd; additionally records events[0..3]
 * (cudaEvent_t handles created by the caller, each may be NULL) on `stream`:
 * [0] before the row-statistics kernel, [1] before the demand sweep, [2]
 * before the finalize kernel, [3] after it.  Used to time each kernel on the
 * stream it runs on.  events == NULL is the same as dilution_attn_fwd. */
int dilution_attn_fwd_with_events(const void *q, const void *k, const void *v, void *out,
                                  float *lse2_out, float *rowsum_out, float *demand_out,
                                  int B, int H, int T, int d, float tau, float eps, int dtype,
                                  void *workspace, size_t workspace_bytes, void *stream,
                                  void *const *events);

/* ------------------------------------------------------------------------
 * Extended forward: dilution_attn_fwd_with_events plus two options.
 *
 *   tau_bh  nullable DEVICE pointer to B*H fp32 logit multipliers, index
 *           b*H + h: head (b, h) uses tau_bh[b*H + h] instead of `tau` (a
 *           per-head temperature, "Learning to Focus: Focal Attention for
 *           Selective and Scalable Transformers", section "Transformer with
 *           Learned Temperature": learned there, an input here).  4-byte
 *           aligned.  `tau` is still validated but unused when tau_bh is
 *           given.  Entries must be finite and >= 0; the kernels cannot
 *           return a synchronous error for device data, so a negative, NaN or
 *           infinite entry sets DA_ERR_INVALID in the status word
 *           (dilution_attn_get_error) and that head's results are unspecified.
 *           The backward and decode calls of the same model must receive the
 *           same array.
 *   flags   DA_FLAG_EARLIER_DEMAND_ONLY: the ablation of "DilutionAttention
 *           v0.1.0 · results" (paragraph after "The operator") that divides
 *           each bid by the demand of earlier queries alone,
 *               share_ik = p_ik / (committed_ik + eps),
 *           so every key's first query (the key itself) gets share p_ii / eps
 *           and, as eps -> 0, the layer tends to the identity map.  For
 *           DA_BF16, shares up to 1/eps are fed to the value product in bf16;
 *           eps >= 1e-18 as for the default operator.
 *           DA_FLAG_KEEP_FOR_BACKWARD (DA_BF16 only, else DA_ERR_UNSUPPORTED):
 *           the workspace must be at least dilution_attn_bwd_workspace_size()
 *           (else DA_ERR_WORKSPACE); the forward also leaves there what the
 *           backward would otherwise recompute (the demand of every key at
 *           every 32-query chunk and the unnormalised outputs), so that a
 *           dilution_attn_bwd_ex with the same flag, the same inputs,
 *           options and workspace skips that pass.  The caller must not
 *           touch the workspace in between.
 *   events  as for dilution_attn_fwd_with_events (nullable).
 * Other arguments, outputs and errors as for dilution_attn_fwd; unknown flag
 * bits or a misaligned tau_bh return DA_ERR_INVALID.
 * ---------------------------------------------------------------------- */
int dilution_attn_fwd_ex(const void *q, const void *k, const void *v, void *out,
                         float *lse2_out, float *rowsum_out, float *demand_out,
                         int B, int H, int T, int d, float tau, const float *tau_bh, float eps,
                         int flags, int dtype, void *workspace, size_t workspace_bytes, void *stream,
                         void *const *events);

/* ------------------------------------------------------------------------
 * Backward: gradients dq, dk, dv [B,H,T,d] of sum(dout * out) for the
 * forward above (the page states only that exact gradients exist; they are
 * the chain rule through the causal softmax, the exclusive column cumsum, the
 * share and the renormalisation).
 *   lse2 [B,H,T] fp32: the forward's lse2_out for the same q, k, tau.
 *   dtype applies to q, k, v, dout, dq, dk, dv.  DA_BF16 runs on tcgen05
 *   tensor cores (bf16 products, fp32 accumulation and fp32 demand
 *   arithmetic, the demand recomputed from checkpoints every 32 queries; the
 *   products' operands are rounded to bf16: the shares, u = p dp, p rho, ds
 *   and dout divided by each row's sum of shares);
 *   DA_F32 runs on CUDA cores in fp32 (column sums of the demand in fp64).
 * workspace: at least dilution_attn_bwd_workspace_size(); errors as for
 * dilution_attn_fwd.
 * ---------------------------------------------------------------------- */
size_t dilution_attn_bwd_workspace_size(int B, int H, int T, int d, int dtype);

int dilution_attn_bwd(const void *q, const void *k, const void *v, const void *dout,
                      const float *lse2, void *dq, void *dk, void *dv,
                      int B, int H, int T, int d, float tau, float eps, int dtype,
                      void *workspace, size_t workspace_bytes, void *stream);

/* Backward with the options of dilution_attn_fwd_ex: tau_bh (nullable device
 * [B*H]) and flags (DA_FLAG_EARLIER_DEMAND_ONLY), which must match the
 * forward that produced lse2.  DA_FLAG_KEEP_FOR_BACKWARD (DA_BF16 only):
 * workspace is the one the forward ran with under the same flag and still
 * holds its state; lse2 is then not read (but must still be a valid pointer).
 * With DA_FLAG_EARLIER_DEMAND_ONLY, D_jk = committed_jk + eps and the direct
 * term of dp_jk is dr_jk / D_jk.  Errors as for dilution_attn_bwd
 * plus those of dilution_attn_fwd_ex for tau_bh and flags. */
int dilution_attn_bwd_ex(const void *q, const void *k, const void *v, const void *dout,
                         const float *lse2, void *dq, void *dk, void *dv,
                         int B, int H, int T, int d, float tau, const float *tau_bh, float eps,
                         int flags, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Cached decode step ("DilutionAttention v0.1.0 · results", section "The
 * operator": the ordinary key/value cache plus one running demand total per
 * key and head).
 *
 * For each (b, h): the cache holds keys/values 0 .. n_ctx-1 in
 * k_cache/v_cache [B,H,T_cap,d] and their demand totals in demand
 * [B,H,T_cap] (fp32; sum of every bid each key has received so far).  The
 * step
 *   1. writes k_new/v_new [B,H,d] to position n_ctx of the caches,
 *   2. forms the bids p_k of q_new [B,H,d] over keys 0 .. n_ctx (causal
 *      softmax of the scaled logits),
 *   3. share_k = p_k / (demand_k + p_k + eps), with demand_{n_ctx} = 0,
 *   4. out [B,H,d] = sum_k share_k v_k / sum_k share_k,
 *   5. demand_k += p_k for k <= n_ctx (in place; demand_{n_ctx} = p_{n_ctx}).
 * Requires 0 <= n_ctx < T_cap.  After the call the cache holds n_ctx + 1
 * tokens.  dtype applies to q/k/v/out and the caches (DA_BF16 only).
 * workspace: at least dilution_attn_decode_workspace_size(B,H,T_cap,d).
 * ---------------------------------------------------------------------- */
size_t dilution_attn_decode_workspace_size(int B, int H, int T_cap, int d);

int dilution_attn_decode_step(const void *q_new, const void *k_new, const void *v_new,
                              void *k_cache, void *v_cache, float *demand,
                              int n_ctx, int T_cap, void *out,
                              int B, int H, int d, float tau, float eps, int dtype,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Decode step with the options of dilution_attn_fwd_ex: tau_bh (nullable
 * device [B*H]) and flags.  With DA_FLAG_EARLIER_DEMAND_ONLY step 3 becomes
 * share_k = p_k / (demand_k + eps); the demand update is unchanged, so a
 * cache built by a flagged prefill continues the flagged operator.  Errors as
 * for dilution_attn_decode_step plus those of dilution_attn_fwd_ex for tau_bh
 * and flags (DA_FLAG_KEEP_FOR_BACKWARD is DA_ERR_INVALID here). */
int dilution_attn_decode_step_ex(const void *q_new, const void *k_new, const void *v_new,
                                 void *k_cache, void *v_cache, float *demand,
                                 int n_ctx, int T_cap, void *out,
                                 int B, int H, int d, float tau, const float *tau_bh, float eps,
                                 int flags, int dtype, void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------------
 * Cached decode step that allocates nothing (no counterpart on the pages: an
 * interface convenience, not part of the method).
 *
 * Same arguments, semantics and errors as dilution_attn_decode_step, without
 * the workspace: scratch comes from a fixed 16 MiB array built into the
 * library (dilution_attn_decode_noalloc_scratch_bytes()).  It is for callers
 * that cannot allocate device memory while decoding -- a runtime whose memory
 * pool is fixed for the duration of a request, or a host that can pass only
 * the tensors it already owns.  Every GPU that loads the library keeps the
 * array until the process exits.
 *   - Returns DA_ERR_WORKSPACE when dilution_attn_decode_workspace_size(B, H,
 *     T_cap, d) exceeds the array (e.g. 8 x 12 heads fit T_cap up to ~42K).
 *   - Calls no cudaMalloc/cudaFree; the first call on a device looks up the
 *     array's device address (cudaGetSymbolAddress), so make that first call
 *     before any stream capture.
 *   - All calls share the array and it keeps the last call's contents (the
 *     status word is cleared at the start of each call): calls that overlap on
 *     the GPU race with each other, so issue them on one stream or order them.
 *   - Errors found on the device (a bounded wait that ran out, an invalid
 *     per-head scale) land in the array's status word: read and clear it with
 *     dilution_attn_decode_noalloc_get_error.
 * ---------------------------------------------------------------------- */
int dilution_attn_decode_step_noalloc(const void *q_new, const void *k_new, const void *v_new,
                                      void *k_cache, void *v_cache, float *demand,
                                      int n_ctx, int T_cap, void *out,
                                      int B, int H, int d, float tau, float eps, int dtype,
                                      void *stream);

/* Size in bytes of the fixed scratch array of dilution_attn_decode_step_noalloc. */
size_t dilution_attn_decode_noalloc_scratch_bytes(void);

/* Synchronises `stream` and returns the status word of the fixed array on the
 * current device (DA_OK, or the first error a kernel of an earlier no-alloc
 * call recorded, e.g. DA_ERR_TIMEOUT), clearing it; DA_ERR_CUDA if the array
 * cannot be reached.  Same semantics as dilution_attn_get_error on a
 * workspace. */
int dilution_attn_decode_noalloc_get_error(void *stream);

/* ------------------------------------------------------------------------
 * Synchronises `stream`, reads the status word that kernels of the last call
 * on `workspace` may have set, clears it and returns it (DA_OK if none).
 * Returns DA_ERR_CUDA if the synchronisation or the copy fails.
 * ---------------------------------------------------------------------- */
int dilution_attn_get_error(void *workspace, void *stream);

/* Copies the workspace's 4-word status block to host `out` after a device
 * synchronisation: [0] status, and when a bounded wait timed out, [1] the
 * shared-memory offset of the mbarrier it waited on, [2] the block index,
 * [3] the thread index of the first wait that gave up.  Diagnostic only. */
int dilution_attn_debug_last_timeout(void *workspace, int32_t *out);

/* ------------------------------------------------------------------------
 * Test hook of the bounded waits (diagnostic only; no counterpart on the
 * pages).  Runs one decode step like dilution_attn_decode_step (same
 * arguments, tau_bh = NULL, flags = 0), except that
 *   - in the first kernel's block for key chunk `stall_chunk` (2048 keys per
 *     chunk) of head stall_bh (= b*H + h), one consumer warp keeps the first
 *     ring stage it read instead of handing it back, so the block's copy
 *     producer waits for a shared-memory slot that is never freed (the chunk
 *     needs at least three 256-key stages of cached keys before n_ctx);
 *   - every wait of that kernel gives up after wait_limit_ns (1e3 .. 1e9 ns).
 * The waits that run out record DA_ERR_TIMEOUT and their place
 * (dilution_attn_debug_last_timeout: status, barrier offset, block index =
 * stall_chunk, thread index) in the workspace status word; the blocks that
 * gave up finish without waiting further, so the call completes and the
 * device stays usable.  The step's outputs, the appended cache row and the
 * demand are then unspecified.  Errors: those of dilution_attn_decode_step,
 * and DA_ERR_INVALID for a wait_limit_ns outside the range, a negative
 * stall_chunk or a stall_bh outside [0, B*H).
 * ---------------------------------------------------------------------- */
int dilution_attn_debug_decode_stall(const void *q_new, const void *k_new, const void *v_new,
                                     void *k_cache, void *v_cache, float *demand,
                                     int n_ctx, int T_cap, void *out,
                                     int B, int H, int d, float tau, float eps, int dtype,
                                     void *workspace, size_t workspace_bytes, void *stream,
                                     int stall_chunk, int stall_bh, long long wait_limit_ns);

/* ------------------------------------------------------------------------
 * Host-only introspection of integer artefacts (no GPU needed).
 *
 * dilution_attn_debug_tile_schedule: the work order of the bf16 forward's and
 * backward's kernels for a problem of BH = B*H heads and T tokens.  kernel = 0 (row
 * statistics at d = 64: pairs of 128-row query tiles, heads in groups of
 * about 96 MB of Q and K), 1 (demand sweep at d = 64: 128-row query tiles,
 * 384-key spans), 2 (demand sweep at d = 128: 256-key spans), 3 (row
 * statistics at d = 128), or 4 + 2 * pass + (d == 128) for the tensor-core
 * backward's passes (pass 0: reverse pass, 1: light dK pass, one CTA per
 * 128-key tile; 2: dQ pass, one CTA per 128-query tile).  For each CTA index
 * c (in launch order), writes 4 int32 to out[4c..4c+3]: head index, first
 * query tile, number of query tiles (row stats: the query tiles it owns;
 * sweep and key-tile passes: the query tiles it walks, from its diagonal; dQ
 * pass: 1, its own), first key (sweep and key-tile passes) or 0.  Returns the number of CTAs; if cap (in
 * int32 elements) is too small, writes nothing and returns -(needed).
 *
 * dilution_attn_debug_tile_mask: the causal mask the kernels apply to the
 * 128 x 128 tile (query tile qt, key tile kt) of a T-token head: out[r*128+c]
 * = 1 if query qt*128+r may see key kt*128+c (key <= query < T), else 0.
 * ---------------------------------------------------------------------- */
int dilution_attn_debug_tile_schedule(int BH, int T, int kernel, int32_t *out, size_t cap);
int dilution_attn_debug_tile_mask(int T, int qt, int kt, uint8_t *out);

#ifdef __cplusplus
}
#endif

#endif /* DILUTION_ATTN_H */
