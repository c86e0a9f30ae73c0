// Internal constants, workspace layout and tile schedules shared by the
// host-side C ABI and the kernels.  Host and device evaluate the same
// schedule functions, so the debug export reproduces the kernels' order.
#pragma once

#include <atomic>
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/dilution_attn.h"

#if defined(__CUDACC__)
#define DA_HD __host__ __device__ __forceinline__
#else
#define DA_HD inline
#endif

namespace da {

// Head dimensions: 64 and 128 (every kernel is instantiated for both).
constexpr int kD = 64;             // the default head dimension
constexpr int kDMax = 128;
constexpr int kTile = 128;         // query / key tile edge (one TMEM lane per row)
constexpr int kSpan = 256;         // Tp granule: two 128-row tiles (one row-statistics CTA)
constexpr size_t kStatusBytes = 256;
// Status block words: [0] status code, [1..3] where a bounded wait gave up,
// [4] rows the row-statistics pass marked for exact recomputation.  Words
// 0..kStatusWordsReset-1 are cleared before every call.
constexpr int kStatusRowsRedo = 4;
constexpr int kStatusWordsReset = 8;

DA_HD bool head_dim_supported(int d) { return d == 64 || d == 128; }
// fp32 per accumulator row: d numerator + row sum + 3 pad (16-byte rows).
DA_HD constexpr int acc_stride(int d) { return d + 4; }
constexpr int kAccStride = acc_stride(kD);

DA_HD int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }
DA_HD int64_t t_pad(int64_t T) { return round_up(T, kSpan); }

// ---------------------------------------------------------------------------
// Workspace of the forward: [status | lse2 [BH][Tp] | acc [BH][Tp][d + 4]].
// Padded rows (T <= row < Tp) carry lse2 = +inf so their bids are exactly 0.
// ---------------------------------------------------------------------------
struct FwdWorkspace {
  size_t lse2_off, acc_off, total;
};

DA_HD FwdWorkspace fwd_workspace_layout(int64_t BH, int64_t T, int d) {
  FwdWorkspace w;
  const int64_t Tp = t_pad(T);
  w.lse2_off = kStatusBytes;
  w.acc_off = (size_t)round_up((int64_t)w.lse2_off + BH * Tp * 4, 256);
  w.total = (size_t)round_up((int64_t)w.acc_off + BH * Tp * acc_stride(d) * 4, 256);
  return w;
}

// ---------------------------------------------------------------------------
// Backward workspace: [status | column totals [BH][T] fp64 | R, Y, rho, spare
// [4][BH][T] fp32 | dq accumulator [BH][T][d] fp32]
// ---------------------------------------------------------------------------
struct BwdWorkspace {
  size_t dtot_off, row_off, dq_off, total;
};

DA_HD BwdWorkspace bwd_workspace_layout(int64_t BH, int64_t T, int d) {
  BwdWorkspace w;
  w.dtot_off = kStatusBytes;
  w.row_off = (size_t)round_up((int64_t)w.dtot_off + BH * T * 8, 256);
  w.dq_off = (size_t)round_up((int64_t)w.row_off + 4 * BH * T * 4, 256);
  w.total = (size_t)round_up((int64_t)w.dq_off + BH * T * d * 4, 256);
  return w;
}

// ---------------------------------------------------------------------------
// Tensor-core backward workspace (bf16):
// [status | -lse2 [BH][Tp] | acc [BH][Tp][d + 4] | delta / R, rho [2][BH][Tp] |
//  demand checkpoints [BH][Tp/32][Tp] | reverse-sum checkpoints [BH][Tp/32][Tp] |
//  dK1 [BH][T][d] fp32 | dout / R [BH][T][d] bf16]
// The checkpoints hold, for every key and every 32-query chunk at or after
// the key's sweep span, committed + eps (forward order) and the sum of dC
// over the queries after the chunk (reverse order).  dK1 is the part of dK
// that the reverse pass accumulates (sum_j p dp q_j, before the scale).
// dout / R (each row of the upstream gradient divided by its row's R) takes
// the place of dout in the tensor-core products, so they give dr and dV
// without a 1/R factor per pair.
// ---------------------------------------------------------------------------
struct BwdTcWorkspace {
  size_t nlse2_off, acc_off, rows_off, cchk_off, gchk_off, dk1_off, gs_off, total;
};

DA_HD BwdTcWorkspace bwd_tc_workspace_layout(int64_t BH, int64_t T, int d) {
  BwdTcWorkspace w;
  const int64_t Tp = t_pad(T);
  w.nlse2_off = kStatusBytes;
  w.acc_off = (size_t)round_up((int64_t)w.nlse2_off + BH * Tp * 4, 256);
  w.rows_off = (size_t)round_up((int64_t)w.acc_off + BH * Tp * acc_stride(d) * 4, 256);
  w.cchk_off = (size_t)round_up((int64_t)w.rows_off + 2 * BH * Tp * 4, 256);
  w.gchk_off = (size_t)round_up((int64_t)w.cchk_off + BH * (Tp / 32) * Tp * 4, 256);
  w.dk1_off = (size_t)round_up((int64_t)w.gchk_off + BH * (Tp / 32) * Tp * 4, 256);
  w.gs_off = (size_t)round_up((int64_t)w.dk1_off + BH * T * d * 4, 256);
  w.total = (size_t)round_up((int64_t)w.gs_off + BH * T * d * 2, 256);
  return w;
}

// ---------------------------------------------------------------------------
// Decode workspace: [status | logits [BH][T_cap] | part_ml [BH][nchunk][2] |
//                    part_acc [BH][nchunk][d + 4]]
// ---------------------------------------------------------------------------
constexpr int kDecChunk = 2048;    // keys per decode CTA (measured: 2048 beats 1024 and 4096)

// Test hook of the decode step's bounded waits: in the first kernel's block
// (chunk stall_chunk, head stall_bh), consumer warp 0 keeps its hand-off of
// ring stage 0, so the block's copy producer waits for a slot that is never
// freed; every wait of that kernel gives up after wait_limit_ns.  The
// ordinary step passes stall_chunk = -1 and the 1 s limit.
struct DecDebug {
  unsigned long long wait_limit_ns;
  int stall_chunk, stall_bh;
};

struct DecWorkspace {
  size_t logit_off, ml_off, acc_off, total;
  int nchunk;
};

DA_HD DecWorkspace dec_workspace_layout(int64_t BH, int64_t T_cap, int d) {
  DecWorkspace w;
  w.nchunk = (int)((T_cap + kDecChunk - 1) / kDecChunk);
  w.logit_off = kStatusBytes;
  w.ml_off = (size_t)round_up((int64_t)w.logit_off + BH * T_cap * 4, 256);
  w.acc_off = (size_t)round_up((int64_t)w.ml_off + BH * w.nchunk * 2 * 4, 256);
  w.total = (size_t)round_up((int64_t)w.acc_off + BH * w.nchunk * acc_stride(d) * 4, 256);
  return w;
}

// ---------------------------------------------------------------------------
// Tile schedules (bf16 forward).  Launch order puts the CTAs with the most
// causal work first so the hardware block scheduler approximates
// longest-processing-time-first across the 152 SMs.
// ---------------------------------------------------------------------------
struct TileWork {
  int bh, q_tile0, n_q_tiles, key0;
};

// Launch order shared by the kernels below: heads in groups of hg (a smaller
// remainder group first, so that its longest CTAs do not run alone at the
// end), and inside a group work item i = 0, 1, ... for each head of the group
// in turn (item 0 is the longest).  Returns the head in bh and the item in i.
DA_HD void grouped_order(int cta, int BH, int hg, int items_per_head, int &bh, int &i) {
  const int ngroups = (BH + hg - 1) / hg;
  const int first = BH - (ngroups - 1) * hg;       // heads in group 0 (1 .. hg)
  int h0, ng;
  if (cta < first * items_per_head) {
    h0 = 0;
    ng = first;
  } else {
    h0 = first + (cta - first * items_per_head) / (hg * items_per_head) * hg;
    ng = hg;
  }
  const int r = cta - h0 * items_per_head;
  bh = h0 + r % ng;
  i = r / ng;
}
DA_HD int clamp_group(int64_t hg, int BH) { return (int)(hg < 1 ? 1 : (hg > BH ? BH : hg)); }

// Row statistics: one CTA per pair of query tiles (2 x 128 rows), each
// streaming its head's key tiles from the first to its diagonal.  Heads are
// taken in groups whose Q and K (Tp x d x 2 B each per head) together stay
// near 96 MB, so that the CTAs in flight share their heads' key tiles in L2
// instead of re-reading them from DRAM; inside a group the pairs with the
// most keys launch first, and a smaller remainder group goes first (as in the
// sweep below, so that its long pairs do not run alone at the end).
constexpr int64_t kRsGroupBytes = 96ll << 20;
DA_HD int rowstats_num_ctas(int BH, int64_t T) { return BH * (int)(t_pad(T) / (2 * kTile)); }
DA_HD int rowstats_head_group(int BH, int64_t T, int d) {
  return clamp_group(kRsGroupBytes / (t_pad(T) * d * 4), BH);
}
DA_HD TileWork rowstats_work(int cta, int BH, int64_t T, int d) {
  const int npairs = (int)(t_pad(T) / (2 * kTile));
  int bh, i;
  grouped_order(cta, BH, rowstats_head_group(BH, T, d), npairs, bh, i);
  TileWork w;
  w.bh = bh;
  const int pair = npairs - 1 - i;   // the last pair sees the most keys
  w.q_tile0 = 2 * pair;
  w.n_q_tiles = 2;
  w.key0 = 0;
  return w;
}

// Demand sweep: one CTA per span of keys (three 128-key tiles at d = 64, two
// at d = 128), walking 128-query tiles from the span's first query tile to
// the end.  Heads are taken in groups whose fp32 accumulators (Tp x (d + 4) x
// 4 B per head) together stay near 64 MB, so the reductions of the CTAs in
// flight hit L2; inside a group the spans with the most query tiles launch
// first.  When BH is not a multiple of the group size, the smaller remainder
// group goes FIRST: launched last, its long first spans would start after
// every other group and run alone at the end (4 x 12 x 16384: groups 15, 15,
// 15, 3 leave ~7 % of the SM time idle in a greedy list-scheduling model; 3,
// 15, 15, 15 leave ~0.5 %).
constexpr int kSweepQTile = 128;
constexpr int64_t kAccGroupBytes = 64ll << 20;
DA_HD int sweep_span_keys(int d) { return d == 64 ? 384 : 256; }
DA_HD int sweep_num_spans(int64_t T, int d) {
  return (int)((t_pad(T) + sweep_span_keys(d) - 1) / sweep_span_keys(d));
}
DA_HD int sweep_head_group(int BH, int64_t T, int d) {
  return clamp_group(kAccGroupBytes / (t_pad(T) * acc_stride(d) * 4), BH);
}
DA_HD int sweep_num_ctas(int BH, int64_t T, int d) { return BH * sweep_num_spans(T, d); }
DA_HD TileWork sweep_work(int cta, int BH, int64_t T, int d) {
  const int nqt = (int)(t_pad(T) / kSweepQTile);
  int bh, span;   // span 0 walks every query tile
  grouped_order(cta, BH, sweep_head_group(BH, T, d), sweep_num_spans(T, d), bh, span);
  TileWork w;
  w.bh = bh;
  w.key0 = span * sweep_span_keys(d);
  w.q_tile0 = w.key0 / kSweepQTile;
  w.n_q_tiles = nqt - w.q_tile0;
  return w;
}

// Tensor-core backward: the reverse pass (R) and the light dK pass (L) take
// one CTA per (head, 128-key tile), walking the query half tiles from the
// last one back to the key tile's diagonal (key tile 0 walks the most); the
// dQ pass one CTA per (head, 128-query tile), walking key tiles 0 .. its
// diagonal (the last query tile walks the most).  Heads in groups whose two
// streamed [Tp x d] bf16 operands (R: Q and dout; L: Q and K; dQ pass: K and
// V) total about 96 MB, so that the tiles every CTA of a head streams are
// shared in L2 by the CTAs in flight; R at d = 64 keeps the plain order
// (every head's key tile 0, then every head's key tile 1, ...), which
// measured faster there.
//   R, L:    key0 = first key, q_tile0 = the diagonal query tile,
//            n_q_tiles = query tiles walked;
//   dQ pass: q_tile0 = its query tile, n_q_tiles = 1, key0 = 0.
constexpr int kBwdRev = 0, kBwdDk2 = 1, kBwdDq = 2;
constexpr int64_t kBwdGroupBytes = 96ll << 20;
DA_HD int bwd_num_ctas(int BH, int64_t T) { return BH * (int)(t_pad(T) / kTile); }
DA_HD int bwd_head_group(int BH, int64_t T, int d) { return clamp_group(kBwdGroupBytes / (t_pad(T) * d * 4), BH); }
DA_HD TileWork bwd_work(int cta, int BH, int64_t T, int d, int pass) {
  const int nt = (int)(t_pad(T) / kTile);
  int bh, i;
  if (pass == kBwdRev && d == 64) {
    bh = cta % BH;
    i = cta / BH;
  } else {
    grouped_order(cta, BH, bwd_head_group(BH, T, d), nt, bh, i);
  }
  TileWork w;
  w.bh = bh;
  if (pass == kBwdDq) {
    w.q_tile0 = nt - 1 - i;
    w.n_q_tiles = 1;
    w.key0 = 0;
  } else {
    w.key0 = i * kTile;
    w.q_tile0 = i;
    w.n_q_tiles = nt - i;
  }
  return w;
}

// ---------------------------------------------------------------------------
// Logit scale of one (batch, head) in the log2 domain, c2 = tau log2(e) /
// sqrt(d).  tau_bh (device [BH], nullable) holds one multiplier per head;
// without it every head uses the scalar's c2.  Both are formed in double and
// rounded once, so equal multipliers give bit-identical scales.
// ---------------------------------------------------------------------------
struct HeadScale {
  const float *tau_bh;
  float c2;        // scalar tau * log2(e) / sqrt(d)
  double per_tau;  // log2(e) / sqrt(d)
};

#if defined(__CUDACC__)
// A negative, NaN or infinite entry records DA_ERR_INVALID in the status word
// (when given) and yields 0, i.e. uniform bids.
__device__ __forceinline__ float head_c2(const HeadScale &hs, int bh, int *status) {
  if (hs.tau_bh == nullptr) return hs.c2;
  const float t = __ldg(hs.tau_bh + bh);
  if (!(t >= 0.f && t <= 3.0e38f)) {
    if (status != nullptr) atomicCAS(status, DA_OK, DA_ERR_INVALID);
    return 0.f;
  }
  return (float)((double)t * hs.per_tau);   // rounded once, as the scalar's c2
}
#endif

// One-time set-up per device (function attributes such as the shared-memory
// opt-in are per device).  Several host threads may make their first call on
// a device at the same time: the set-up runs under a lock, once, and later
// calls see the flag without locking.  `setup` returns a da status; a failed
// set-up is retried by the next call.  Devices past the table's 64 entries
// run the set-up on every call.
struct PerDeviceOnce {
  std::mutex mu;
  std::atomic<bool> done[64] = {};

  template <typename F>
  int run(F &&setup) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DA_ERR_CUDA;
    if (dev < 0 || dev >= 64) return setup();
    if (done[dev].load(std::memory_order_acquire)) return DA_OK;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev].load(std::memory_order_relaxed)) return DA_OK;
    const int st = setup();
    if (st == DA_OK) done[dev].store(true, std::memory_order_release);
    return st;
  }
};

// Causal mask predicate used by every kernel: query i sees key k iff k <= i
// and i < T ("DilutionAttention v0.1.0 · results", section "The operator":
// causal softmax, diagonal included).
DA_HD bool visible(int64_t i, int64_t k, int64_t T) { return k <= i && i < T; }

}  // namespace da
