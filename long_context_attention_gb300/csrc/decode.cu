// Cached decode step of dilution attention ("DilutionAttention v0.1.0 ·
// results", section "The operator": the key/value cache plus one running
// demand total per key and head).
//
// A share needs the new query's softmax normaliser before it can be formed,
// so the step has two streaming phases separated by kernel boundaries (no
// cross-CTA spinning):
//   dec_logits  : x_k = (q . k_k) * tau/sqrt(d) * log2(e) for k <= n_ctx, written
//                 to a logit scratch, plus one (max, sum 2^(x - max)) per chunk.
//                 The chunk holding position n_ctx also appends k_new / v_new.
//   dec_update  : lse2 from the chunk partials; p_k = 2^(x_k - lse2);
//                 share_k = p_k / (D_k + p_k + eps) with D_{n_ctx} = 0
//                 (p_k / (D_k + eps) in the earlier-demand-only variant);
//                 D_k += p_k in place; per-chunk sum_k share_k v_k and sum_k share_k.
//   dec_combine : out = sum of chunk numerators / sum of chunk row sums
//                 (fixed order: deterministic).
// Memory: K and V rows are read once each, streamed into shared memory by
// bulk copies (8 consumer lanes per 128-byte bf16 row read them from there),
// the demand is read and written once; the fp32 logit scratch (4 B per key)
// stays mostly in L2.
#include "da_internal.h"
#include "da_ptx.cuh"

#include <mutex>

#include <cuda_bf16.h>

namespace da {

constexpr int kDecThreads = 256;

template <typename E>
struct Vec16;   // 16 bytes of one row: 8 bf16 or 4 fp32 elements

template <>
struct Vec16<__nv_bfloat16> {
  static constexpr int N = 8;
  static __device__ __forceinline__ void to_float(const uint4 &u, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
};
template <>
struct Vec16<float> {
  static constexpr int N = 4;
  static __device__ __forceinline__ void to_float(const uint4 &u, float *f) {
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
  }
};

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Lanes per row: a row of d elements is 2d bytes (bf16) or 4d bytes (fp32),
// one 16-byte piece per lane.
template <typename E, int D>
constexpr int lanes_per_row() {
  return D / Vec16<E>::N;
}

// Bulk copy global -> shared with an L2 evict-first policy, for rows read
// exactly once: their lines are the first to go, so the logit scratch and the
// demand written by the same step stay in L2.
__device__ __forceinline__ void bulk_load_stream(void *smem_dst, const void *gmem_src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "{\n\t.reg .b64 pol;\n\t"
      "createpolicy.fractional.L2::evict_first.b64 pol, 1.0;\n\t"
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], pol;\n\t}"
      ::"r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(gmem_src)), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Cache rows stream through a ring of shared-memory stages filled by bulk
// asynchronous copies that one producer warp issues, so the bytes in flight
// do not sit in registers (with register-held loads both streaming kernels
// keep too few bytes in flight per SM to reach HBM rate at their occupancy).
// Whole stages go through the ring; a chunk's tail shorter than a stage is
// read directly.  Every wait is bounded: a timeout records DA_ERR_TIMEOUT in
// the status block and the CTA finishes without waiting further.
// Measured on GB300 (8 x 12 caches of 131072, step time): two 32 KB stages
// 0.508 ms, two 16 KB 0.515, three 16 KB 0.526, four 8 KB 0.555, six 8 KB
// 0.608, eight 4 KB 0.762; 512 consumer threads instead of 256 was slower.
// The stages live in dynamic shared memory (dec_ring_smem), the barriers in
// the kernel's static shared memory.
extern __shared__ __align__(128) uint8_t dec_ring_smem[];

template <typename E, int D>
struct DecRing {
  static constexpr int kRowBytes = D * (int)sizeof(E);
  static constexpr int kStageBytes = 32768;
  static constexpr int kStageKeys = kStageBytes / kRowBytes;   // 256 keys for bf16 rows of 64
  static constexpr int kStages = 2;
  static constexpr int kDynSmemBytes = kStages * kStageBytes;
  static constexpr int kConsumerWarps = kDecThreads / 32;
  static constexpr int kThreads = kDecThreads + 32;            // consumers + the producer warp

  uint64_t full[kStages], empty[kStages];
  int abort_word;

  // one thread, before a __syncthreads
  __device__ __forceinline__ void init() {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    abort_word = 0;
    fence_mbar_init();
  }
  __device__ __forceinline__ WaitCtx wait_ctx(int *status, unsigned long long limit_ns = kWaitLimitNs) {
    return WaitCtx{reinterpret_cast<volatile int *>(&abort_word), status, limit_ns};
  }
  // Producer lane: stages 0 .. n_stage - 1 of the rows starting at `rows`.
  __device__ __forceinline__ void produce(const E *rows, int n_stage, const WaitCtx &wc) {
    int issued = 0;
    for (int st = 0; st < n_stage; ++st) {
      const int s = st % kStages;
      if (!mbar_wait(&empty[s], ((st / kStages) & 1) ^ 1, wc)) break;
      mbar_arrive_expect_tx(&full[s], kStageBytes);
      bulk_load_stream(dec_ring_smem + s * kStageBytes, rows + (size_t)st * kStageKeys * D, kStageBytes, &full[s]);
      ++issued;
    }
    if (abort_word) {   // let the copies in flight land before the CTA exits
      for (int st = (issued > kStages ? issued - kStages : 0); st < issued; ++st) {
        const unsigned long long t0 = globaltimer();
        while (!mbar_try_wait(&full[st % kStages], (st / kStages) & 1))
          if (globaltimer() - t0 > 100ull * 1000ull * 1000ull) break;
      }
    }
  }
  // Consumer warp: wait until stage st has landed (same outcome in every
  // lane, so shuffles may follow), read it, then hand its slot back.
  __device__ __forceinline__ bool ready(int st, const WaitCtx &wc) {
    return warp_wait(&full[st % kStages], (st / kStages) & 1, wc);
  }
  __device__ __forceinline__ const uint8_t *slot(int st) const { return dec_ring_smem + (st % kStages) * kStageBytes; }
  // keep = true (the test hook only): the warp does not hand the slot back.
  __device__ __forceinline__ void release(int st, int lane, bool keep = false) {
    __syncwarp();
    if (lane == 0 && !keep) mbar_arrive(&empty[st % kStages]);
  }
};

template <typename E, int D>
__global__ void __launch_bounds__(DecRing<E, D>::kThreads)
    dec_logits(const E *__restrict__ q_new, const E *__restrict__ k_new, const E *__restrict__ v_new,
               E *__restrict__ k_cache, E *__restrict__ v_cache, float *__restrict__ logits,
               float2 *__restrict__ part_ml, int n_ctx, int T_cap, int nchunk, HeadScale hs, int *status,
               DecDebug dbg) {
  using R = DecRing<E, D>;
  constexpr int LPR = lanes_per_row<E, D>();       // lanes cooperating on one key
  constexpr int NV = Vec16<E>::N;
  constexpr int KPR = kDecThreads / LPR;           // keys per round of the consumers
  constexpr int SK = R::kStageKeys, RPS = SK / KPR;
  static_assert(SK % KPR == 0, "stage of whole rounds");
  const int bh = blockIdx.y, chunk = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const bool producer = warp == R::kConsumerWarps;
  __shared__ R ring;
  const float c2 = head_c2(hs, bh, (tid == 0 && chunk == 0) ? status : nullptr);
  const int sub = tid % LPR;                       // which 16-byte piece of the row
  const int grp = tid / LPR;
  const int k_begin = chunk * kDecChunk;
  const int k_end = min(k_begin + kDecChunk, n_ctx + 1);
  // Whole stages of cached rows before n_ctx go through the ring; key n_ctx
  // (taken from k_new) and the rest of the chunk are read directly.
  const int n_stage = (min(k_end, n_ctx) - k_begin) / SK;
  const E *kb = k_cache + (size_t)bh * T_cap * D;
  if (tid == 0) ring.init();
  __syncthreads();
  const WaitCtx wc = ring.wait_ctx(status, dbg.wait_limit_ns);
  const bool stall = warp == 0 && chunk == dbg.stall_chunk && bh == dbg.stall_bh;   // test hook
  float m = -INFINITY, l = 0.f;
  if (producer) {
    if (lane == 0) ring.produce(kb + (size_t)k_begin * D, n_stage, wc);
  } else {
    float qf[NV];
    Vec16<E>::to_float(*reinterpret_cast<const uint4 *>(q_new + (size_t)bh * D + sub * NV), qf);
    // One key per lane group; every lane of the warp runs it (shuffles), and
    // a key past the chunk (ok = false) leaves the statistics alone.
    auto consume = [&](int key, const uint4 &raw, bool ok) {
      float kf[NV];
      Vec16<E>::to_float(raw, kf);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < NV; ++i) s = fmaf(qf[i], kf[i], s);
#pragma unroll
      for (int off = LPR / 2; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
      if (ok) {
        const float x = s * c2;
        if (sub == 0) logits[(size_t)bh * T_cap + key] = x;
        if (x > m) {
          l = l * exp2f(m - x) + 1.f;
          m = x;
        } else {
          l += exp2f(x - m);
        }
      }
    };
    for (int st = 0; st < n_stage; ++st) {
      if (!ring.ready(st, wc)) break;
      const uint8_t *stg = ring.slot(st);
#pragma unroll
      for (int r = 0; r < RPS; ++r) {
        const int kl = r * KPR + grp;
        consume(k_begin + st * SK + kl, *reinterpret_cast<const uint4 *>(stg + kl * R::kRowBytes + sub * 16), true);
      }
      ring.release(st, lane, stall && st == 0);
    }
    // the tail, with a warp-uniform trip count
    for (int r0 = k_begin + n_stage * SK; r0 < k_end; r0 += KPR) {
      const int key = r0 + grp;
      const bool ok = key < k_end;
      uint4 raw = make_uint4(0u, 0u, 0u, 0u);
      if (ok) raw = ld_stream(((key == n_ctx) ? k_new + (size_t)bh * D : kb + (size_t)key * D) + sub * NV);
      consume(key, raw, ok);
    }
  }
  // Append the new key/value at position n_ctx (done by the chunk holding it).
  if (n_ctx >= k_begin && n_ctx < k_begin + kDecChunk && tid < 2 * LPR) {
    const E *src = (tid < LPR) ? k_new : v_new;
    E *dst = (tid < LPR) ? k_cache : v_cache;
    const int piece = tid % LPR;
    *reinterpret_cast<uint4 *>(dst + ((size_t)bh * T_cap + n_ctx) * D + piece * NV) =
        *reinterpret_cast<const uint4 *>(src + (size_t)bh * D + piece * NV);
  }
  // Block reduction of (m, l): only lane sub == 0 of each consumer group holds data.
  __shared__ float sm[kDecThreads], sl[kDecThreads];
  if (tid < kDecThreads) {
    sm[tid] = (sub == 0) ? m : -INFINITY;
    sl[tid] = (sub == 0) ? l : 0.f;
  }
  __syncthreads();
  for (int stride = kDecThreads / 2; stride > 0; stride >>= 1) {
    if (tid < stride) {
      const float m1 = sm[tid], m2 = sm[tid + stride];
      const float mx = fmaxf(m1, m2);
      float ls = 0.f;
      if (mx != -INFINITY) ls = sl[tid] * exp2f(m1 - mx) + sl[tid + stride] * exp2f(m2 - mx);
      sm[tid] = mx;
      sl[tid] = ls;
    }
    __syncthreads();
  }
  if (tid == 0) part_ml[(size_t)bh * nchunk + chunk] = make_float2(sm[0], sl[0]);
}

template <typename E, int D>
__global__ void __launch_bounds__(DecRing<E, D>::kThreads)
    dec_update(const E *__restrict__ v_cache, const float *__restrict__ logits, const float2 *__restrict__ part_ml,
               float *__restrict__ demand, float *__restrict__ part_acc, int n_ctx, int T_cap, int nchunk,
               int nchunk_used, float eps, bool earlier, int *status) {
  using R = DecRing<E, D>;
  constexpr int LPR = lanes_per_row<E, D>();
  constexpr int NV = Vec16<E>::N;
  constexpr int KPR = kDecThreads / LPR;                // keys per round of the consumers
  constexpr int SK = R::kStageKeys, RPS = SK / KPR;     // rounds per stage
  static_assert(SK % KPR == 0, "stage of whole rounds");
  const int bh = blockIdx.y, chunk = blockIdx.x;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const bool producer = warp == R::kConsumerWarps;
  const int sub = tid % LPR, grp = tid / LPR;
  __shared__ R ring;
  __shared__ float s_lse2;
  const int k_begin = chunk * kDecChunk;
  const int k_end = min(k_begin + kDecChunk, n_ctx + 1);
  const int n_stage = (k_end - k_begin) / SK;           // whole stages through the ring
  const E *vb = v_cache + (size_t)bh * T_cap * D;
  if (tid == 0) ring.init();
  if (tid < 32) {
    // Combine the per-chunk (max, sum) pairs of this head into lse2.
    float m = -INFINITY, l = 0.f;
    for (int c = tid; c < nchunk_used; c += 32) {
      const float2 ml = part_ml[(size_t)bh * nchunk + c];
      if (ml.x == -INFINITY) continue;
      const float mx = fmaxf(m, ml.x);
      l = l * exp2f(m - mx) + ml.y * exp2f(ml.x - mx);
      m = mx;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
      const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
      const float mx = fmaxf(m, m2);
      if (mx != -INFINITY) {
        l = l * exp2f(m - mx) + l2 * exp2f(m2 - mx);
        m = mx;
      }
    }
    if (tid == 0) s_lse2 = m + log2f(l);
  }
  __syncthreads();
  const float lse2 = s_lse2;
  const WaitCtx wc = ring.wait_ctx(status);
  float num[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) num[i] = 0.f;
  float rs = 0.f;

  // one key: its bid, share against the demand, demand update, share * v
  auto consume = [&](int key, const uint4 &raw, float x, float dm) {
    const float p = exp2f(x - lse2);
    const float den = (earlier ? dm : dm + p) + eps;
    const float share = p / den;
    if (sub == 0) demand[(size_t)bh * T_cap + key] = dm + p;
    float vf[NV];
    Vec16<E>::to_float(raw, vf);
#pragma unroll
    for (int i = 0; i < NV; ++i) num[i] = fmaf(share, vf[i], num[i]);
    rs += share;
  };

  if (producer) {
    if (lane == 0) ring.produce(vb + (size_t)k_begin * D, n_stage, wc);
  } else {
    // logits and demand of this thread's keys, one stage ahead
    float xn[RPS], dn[RPS];
    auto fetch = [&](int st, float (&x)[RPS], float (&d)[RPS]) {
#pragma unroll
      for (int r = 0; r < RPS; ++r) {
        const int key = k_begin + st * SK + r * KPR + grp;
        x[r] = logits[(size_t)bh * T_cap + key];
        d[r] = key < n_ctx ? demand[(size_t)bh * T_cap + key] : 0.f;
      }
    };
    if (n_stage > 0) fetch(0, xn, dn);
    for (int st = 0; st < n_stage; ++st) {
      float xc[RPS], dc[RPS];
#pragma unroll
      for (int r = 0; r < RPS; ++r) {
        xc[r] = xn[r];
        dc[r] = dn[r];
      }
      if (st + 1 < n_stage) fetch(st + 1, xn, dn);
      if (!ring.ready(st, wc)) break;
      const uint8_t *stg = ring.slot(st);
#pragma unroll
      for (int r = 0; r < RPS; ++r) {
        const int kl = r * KPR + grp;
        const uint4 raw = *reinterpret_cast<const uint4 *>(stg + kl * R::kRowBytes + sub * 16);
        consume(k_begin + st * SK + kl, raw, xc[r], dc[r]);
      }
      ring.release(st, lane);
    }
    // the tail of the chunk, read directly
    for (int key = k_begin + n_stage * SK + grp; key < k_end; key += KPR) {
      const uint4 raw = ld_stream(vb + (size_t)key * D + sub * NV);
      consume(key, raw, logits[(size_t)bh * T_cap + key], key < n_ctx ? demand[(size_t)bh * T_cap + key] : 0.f);
    }
  }
  // Reduce the KPR key groups: partial rows [KPR][d + 1] in shared memory.
  __shared__ float sacc[KPR][D + 1];
  if (!producer) {
#pragma unroll
    for (int i = 0; i < NV; ++i) sacc[grp][sub * NV + i] = num[i];
    if (sub == 0) sacc[grp][D] = rs;
  }
  __syncthreads();
  if (tid <= D) {
    float a = 0.f;
    for (int gi = 0; gi < KPR; ++gi) a += sacc[gi][tid];
    part_acc[((size_t)bh * nchunk + chunk) * acc_stride(D) + tid] = a;
  }
}

template <typename E, int D>
__global__ void dec_combine(const float *__restrict__ part_acc, E *__restrict__ out, int nchunk, int nchunk_used) {
  const int bh = blockIdx.x;
  const int t = threadIdx.x;   // 0..63
  float a = 0.f, rs = 0.f;
  for (int c = 0; c < nchunk_used; ++c) {
    const float *pa = part_acc + ((size_t)bh * nchunk + c) * acc_stride(D);
    a += pa[t];
    rs += pa[D];
  }
  const float o = a / rs;
  if constexpr (sizeof(E) == 4) {
    out[(size_t)bh * D + t] = o;
  } else {
    out[(size_t)bh * D + t] = __float2bfloat16_rn(o);
  }
}

template <typename E, int D>
static cudaError_t launch_decode_t(const void *q_new, const void *k_new, const void *v_new, void *k_cache,
                                   void *v_cache, float *demand, int n_ctx, int T_cap, void *out, int BH,
                                   HeadScale hs, float eps, bool earlier, float *logits, float2 *part_ml,
                                   float *part_acc, int nchunk, int *status, DecDebug dbg, cudaStream_t stream) {
  using R = DecRing<E, D>;
  // The ring's shared-memory opt-in is a per-device function attribute.
  static PerDeviceOnce once;
  const int prep = once.run([] {
    return (cudaFuncSetAttribute(dec_logits<E, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, R::kDynSmemBytes) !=
                cudaSuccess ||
            cudaFuncSetAttribute(dec_update<E, D>, cudaFuncAttributeMaxDynamicSharedMemorySize, R::kDynSmemBytes) !=
                cudaSuccess)
               ? DA_ERR_CUDA
               : DA_OK;
  });
  if (prep != DA_OK) return cudaErrorInvalidDeviceFunction;
  const int used = (n_ctx + 1 + kDecChunk - 1) / kDecChunk;
  dec_logits<E, D><<<dim3(used, BH), R::kThreads, R::kDynSmemBytes, stream>>>(
      (const E *)q_new, (const E *)k_new, (const E *)v_new, (E *)k_cache, (E *)v_cache, logits, part_ml, n_ctx,
      T_cap, nchunk, hs, status, dbg);
  dec_update<E, D><<<dim3(used, BH), R::kThreads, R::kDynSmemBytes, stream>>>(
      (const E *)v_cache, logits, part_ml, demand, part_acc, n_ctx, T_cap, nchunk, used, eps, earlier, status);
  dec_combine<E, D><<<BH, D, 0, stream>>>(part_acc, (E *)out, nchunk, used);
  return cudaGetLastError();
}

int check_decode_step_args(const void *q_new, const void *k_new, const void *v_new, const void *k_cache,
                           const void *v_cache, const float *demand, int n_ctx, int T_cap, const void *out, int B,
                           int H, int d, float tau, const float *tau_bh, float eps, int flags, int dtype);

cudaError_t launch_decode(const void *q_new, const void *k_new, const void *v_new, void *k_cache, void *v_cache,
                          float *demand, int n_ctx, int T_cap, void *out, int BH, int d, HeadScale hs, float eps,
                          bool earlier, int dtype, float *logits, float2 *part_ml, float *part_acc, int nchunk,
                          int *status, DecDebug dbg, cudaStream_t stream) {
#define DA_DECODE_ARGS                                                                                          \
  q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx, T_cap, out, BH, hs, eps, earlier, logits, part_ml, part_acc, \
      nchunk, status, dbg, stream
  if (dtype == DA_BF16)
    return d == 128 ? launch_decode_t<__nv_bfloat16, 128>(DA_DECODE_ARGS)
                    : launch_decode_t<__nv_bfloat16, 64>(DA_DECODE_ARGS);
  return d == 128 ? launch_decode_t<float, 128>(DA_DECODE_ARGS) : launch_decode_t<float, 64>(DA_DECODE_ARGS);
#undef DA_DECODE_ARGS
}

// ---------------------------------------------------------------------------
// Decode step without a caller workspace.
//
// Some callers cannot allocate device memory at the point where they decode:
// a runtime that owns a fixed memory pool and forbids allocation during a
// request, a foreign host (another language's runtime, a plugin) that can hand
// over only the tensors it already has, or code that must not allocate between
// decode steps.  For them the scratch lives in this fixed array, which every
// GPU that loads the library holds until the process exits.
// ---------------------------------------------------------------------------
constexpr size_t kNoAllocScratchBytes = 16u << 20;   // 16 MiB
static __device__ __align__(256) uint8_t g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch on the current device, looked up once per
// device (the array's name in host code is only a host-side handle).
static int noalloc_scratch(void **ptr) {
  static std::mutex mu;
  static void *addr[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) return DA_ERR_CUDA;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return DA_OK;
}

}  // namespace da

extern "C" int dilution_attn_decode_step_noalloc(const void *q_new, const void *k_new, const void *v_new,
                                                 void *k_cache, void *v_cache, float *demand, int n_ctx, int T_cap,
                                                 void *out, int B, int H, int d, float tau, float eps, int dtype,
                                                 void *stream) {
  using namespace da;
  // The ordinary step's argument checks come first, so a bad argument is
  // reported as such whatever the size; then the size against the array.
  const int chk = check_decode_step_args(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx, T_cap, out, B, H, d,
                                         tau, nullptr, eps, 0, dtype);
  if (chk != DA_OK) return chk;
  const DecWorkspace L = dec_workspace_layout((int64_t)B * H, T_cap, d);
  if (L.total > kNoAllocScratchBytes) return DA_ERR_WORKSPACE;   // beyond the fixed scratch
  void *scratch = nullptr;
  const int st = noalloc_scratch(&scratch);
  if (st != DA_OK) return st;
  // The argument checks, the status-word reset and the launches are the
  // ordinary decode step's, given the fixed array as its workspace.
  return dilution_attn_decode_step(q_new, k_new, v_new, k_cache, v_cache, demand, n_ctx, T_cap, out, B, H, d, tau,
                                   eps, dtype, scratch, kNoAllocScratchBytes, stream);
}

extern "C" size_t dilution_attn_decode_noalloc_scratch_bytes(void) { return da::kNoAllocScratchBytes; }

// The status word of the fixed array (its first word, as in a workspace):
// read and cleared like dilution_attn_get_error's.
extern "C" int dilution_attn_decode_noalloc_get_error(void *stream) {
  void *scratch = nullptr;
  const int st = da::noalloc_scratch(&scratch);
  if (st != DA_OK) return st;
  return dilution_attn_get_error(scratch, stream);
}
