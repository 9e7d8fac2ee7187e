// Exact backward of two-copy block-diffusion attention, for sm_103a.
//
// For every allowed (query, key) pair: P = exp(scale q.k - LSE_q),
// dV += P dO, dP = dO.v, dS = P (dP - D_q) with D_q = rowsum(dO o O),
// dK += scale dS q, dQ += scale dS k.  Clean dK/dV collect contributions of
// clean queries (same or later block) and corrupted queries (later blocks);
// corrupted dK/dV only those of their own block ("CSBP 完全拆解" blog, section
// "CSBP：BP 管损坏块，CP 管干净上下文", backward paragraph: corrupted gradients stay
// with the block owner, clean dK/dV are summed for the clean-shard owner).
//
// One CTA owns one 128-row key tile of one (batch, KV head) and walks every
// (query head of the GQA group, 128-row query tile) its work-list task lists,
// so dK/dV accumulate in TMEM for the whole group and are written once.  Each
// step handles one query tile with N = 128 MMAs throughout; the two compute
// warpgroups take its two 64-column halves in parallel.  Roles (384 threads):
//   warp 0 lane 0  TMA producer: K, V once; per step Q (2 stages) with its LSE
//                  and D slices
//   warp 2 lane 0  TMA producer: dO (one stage for d = 128, refilled while
//                  the dK, dQ^T and S^T MMAs run; two for d = 64)
//   warp 1 lane 0  MMA issuer (it polls its barriers, so a completed MMA
//                  group or a compute-warp arrival is seen at once), per
//                  step i:
//                    dV += P_i^T dO_i        (P^T read from TMEM)
//                    dQ_i^T = K^T dS_i^T; dK += dS_i^T Q_i   (dS^T from smem;
//                    dQ^T first: the compute warps wait on it, not on dK)
//                    S^T_{i+1} = K Q_{i+1}^T; dP^T_{i+1} = V dO_{i+1}^T
//   warps 4..7 / 8..11  compute halves 0 / 1 (query columns 64h..64h+63):
//                  thread t owns key row t (TMEM lane t).  It turns S^T into
//                  P^T (bf16 pairs written back over its S^T columns) and dP^T
//                  into dS^T (bf16, into its 64-column box of a 128B-swizzled
//                  shared tile: the K-major A operand of dK and the MN-major B
//                  operand of dQ^T).  Then it copies its half of dQ^T
//                  (thread t = head-dim row t) out of TMEM, stages its 64
//                  query rows (32 in its dS^T box, 32 in a buffer of its
//                  own) and adds them into the fp32 dQ accumulator with TMA
//                  bulk reduce-adds.
// TMEM columns: S^T (then P^T) at 0, dP^T (then dQ^T) at 128, dV at 256,
// dK at 256 + d.  For d = 64 the dQ^T MMA runs with M = 128 and the upper 64
// rows of K^T read a zero tile.  All shared state lives in the dynamic
// shared-memory window, which must start 1024-byte aligned.
#include <cuda.h>
#include <cuda_runtime.h>

#include "csbp_internal.h"
#include "device_once.h"
#include "mbar_spin.cuh"
#include "pair_math.cuh"
#include "ptx_sm100.cuh"
#include "work_checks.cuh"

namespace csbp {

namespace {

constexpr int kThreads = 384;
constexpr int kHalf = 64;         // query columns per compute warpgroup
constexpr int kStages = 2;        // Q ring depth
constexpr float kLog2e = 1.4426950408889634f;

enum BwdBar {
  C_KV_FULL = 0,
  C_Q_FULL,                         // [kStages]
  C_Q_EMPTY = C_Q_FULL + kStages,   // [kStages]
  C_DO_FULL = C_Q_EMPTY + kStages,  // [kStages]
  C_DO_EMPTY = C_DO_FULL + kStages,  // [up to kStages]
  C_S_FULL = C_DO_EMPTY + kStages,
  C_DP_FULL,
  C_P_READY,
  C_PV_DONE,
  C_DS_READY,
  C_DQ_FULL,
  C_DQ_FREE,
  C_STAGE_FULL,                     // [2] per half: dQ rows staged
  C_X_FREE = C_STAGE_FULL + 2,      // [2] per half: dS^T box read by its reduce-add
  C_SQ_FREE = C_X_FREE + 2,         // [2] per half: staging buffer read by its reduce-add
  C_ACC_DONE = C_SQ_FREE + 2,
  C_DK_DONE,                        // dK_i complete: the dS^T boxes are free
  C_DRAIN,
  C_COUNT
};

template <int D>
struct BwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;   // a 128-row bf16 tile (K, V, Q, dO)
  static constexpr int kBox = kTile * 128;           // one 64-column box of such a tile
  static constexpr int kXBox = kTile * kHalf * 2;    // dS^T box of one half (16 KB)
  // dQ rows of a half (64 x d fp32) are staged partly in its dS^T box, the
  // rest in a buffer of its own; for d = 128 that buffer comes from keeping a
  // single dO stage, whose refill has the dK, dQ^T and S^T MMAs to land.
  static constexpr int kDOStages = (D == 128) ? 1 : 2;
  static constexpr int kRowsX = kXBox / (D * 4);     // dQ rows staged in the dS^T box
  static constexpr int kRowsSQ = kHalf - kRowsX;     // dQ rows staged in the own buffer
  static_assert(kRowsX <= kHalf && kDOStages <= kStages, "staging split");
  static constexpr int kStatBytes = 2 * kTile * 4;   // LSE and D of one query tile
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kZero = kV + kTileBytes;      // zero K^T rows (d = 64 only)
  static constexpr int kQ = kZero + (D == 64 ? kBox : 0);
  static constexpr int kDO = kQ + kStages * kTileBytes;
  static constexpr int kX = kDO + kDOStages * kTileBytes;
  static constexpr int kSQ = kX + 2 * kXBox;          // [2 halves][kRowsSQ][D] fp32
  static constexpr int kStat = kSQ + 2 * kRowsSQ * D * 4;
  static constexpr int kBar = kStat + kStages * kStatBytes;
  static constexpr int kMisc = kBar + C_COUNT * 8;   // tmem base, abort flag
  static constexpr int kBytes = kMisc + 16;
  static constexpr int kDynSmem = kBytes;            // window is 1024-aligned
  static constexpr uint32_t kColS = 0;
  static constexpr uint32_t kColDP = 128;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
};

// Walk over the (query tile, segment, query head in group) steps of a task:
// query tiles in some order, every segment (query stream) that holds the
// tile, then the heads of the GQA group.
//  - Default: from the last tile down.  Every key tile of a stream is read by
//    the last query tiles, so CTAs that start together stay on the same query
//    tile, and their dQ reduce-adds and Q / dO loads of that tile meet in L2.
//  - Modular (sliding-window masks): the task's tiles span lo .. lo + n - 1
//    and step tau visits the one that is congruent to -tau mod n.  Key tile k
//    is read by query tiles k .. k + n - 1 for a fixed n, so at step tau the
//    CTAs of a wave all visit tiles of one residue class, and a query tile's
//    n readers take it in the same step rather than n steps apart.
struct QWalk {
  const int32_t* seg0;
  int n_segs, G, g, si, t, stream, flags;
  int lo, n, tau;  // modular order (n > 0)
  __device__ bool holds(int s, int tile) const {
    const int32_t* x = seg0 + s * kSegWords;
    return x[1] <= tile && tile < x[2];
  }
  __device__ int find(int from) const {  // first segment >= from holding t
    int s = from;
    while (s < n_segs && !holds(s, t)) ++s;
    return s;
  }
  __device__ void load_seg() {
    const int32_t* x = seg0 + si * kSegWords;
    stream = x[0];
    flags = x[3];
  }
  __device__ int mod_tile(int k) const {  // tile of modular step k
    const int r = ((-k - lo) % n + n) % n;
    return lo + r;
  }
  __device__ void start(const int32_t* s, int n_seg, int group, bool modular) {
    seg0 = s;
    n_segs = n_seg;
    G = group;
    g = 0;
    t = -1;
    lo = 0x7fffffff;
    n = 0;
    tau = 0;
    for (int k = 0; k < n_seg; ++k) {
      t = max(t, s[k * kSegWords + 2] - 1);
      lo = min(lo, s[k * kSegWords + 1]);
    }
    if (modular && t >= lo) {
      n = t - lo + 1;
      t = mod_tile(0);
      si = find(0);
      while (si >= n_segs && ++tau < n) {
        t = mod_tile(tau);
        si = find(0);
      }
    } else {
      si = find(0);
    }
    if (si < n_segs) load_seg();
  }
  __device__ void next() {
    if (++g < G) return;
    g = 0;
    si = find(si + 1);
    if (n > 0) {
      while (si >= n_segs && ++tau < n) {
        t = mod_tile(tau);
        si = find(0);
      }
    } else {
      while (si >= n_segs && t > 0) {
        --t;
        si = find(0);
      }
    }
    if (si < n_segs) load_seg();
  }
};

// Query positions [lo, hi) of copy q_stream that may read key position kpos
// (block kb) of copy k_stream: clean keys are read by clean queries of the
// same or later blocks (queries >= kpos when token-causal) and by corrupted
// queries of later blocks; corrupted keys only by corrupted queries of their
// own block; a window W > 0 also drops queries W or more positions after.
__device__ __forceinline__ void allowed_query_range(int q_stream, int k_stream, int kpos, int kb,
                                                    int M, int L, int window, int clean_causal,
                                                    bool k_valid, int& lo, int& hi) {
  if (!k_valid || (q_stream == 0 && k_stream == 1)) {
    lo = hi = 0;
    return;
  }
  if (k_stream == 0) {
    lo = (q_stream == 0) ? (clean_causal ? kpos : kb * M) : (kb + 1) * M;
    hi = L;
  } else {
    lo = kb * M;
    hi = min((kb + 1) * M, L);
  }
  if (window > 0) hi = min(hi, kpos + window);
}

// P^T of two query columns: 2^(s scale log2e - LSE log2e), the two
// exponent arguments formed in one packed instruction each step.
__device__ __forceinline__ void p_exp2(float s0, float s1, float2 lse, uint64_t sl2x2, float& e0,
                                       float& e1) {
  const uint64_t nl = f2_mul(f2_pack(lse.x, lse.y), f2_pack(-kLog2e, -kLog2e));
  float x0, x1;
  f2_unpack(f2_fma(f2_pack(s0, s1), sl2x2, nl), x0, x1);
  e0 = ex2_approx(x0);
  e1 = ex2_approx(x1);
}

// dS^T = P^T o (dP^T - D) of two query columns, as a bf16 pair.
__device__ __forceinline__ uint32_t ds_pair(float p0, float p1, float dp0, float dp1, float2 dq) {
  float a, b;
  f2_unpack(f2_mul(f2_pack(p0, p1), f2_sub(f2_pack(dp0, dp1), f2_pack(dq.x, dq.y))), a, b);
  return pack_bf16x2(a, b);
}

// S^T (or dP^T) of one step: M = 128 key rows, N = 128 query rows, K = d.
template <int D>
__device__ __forceinline__ void issue_kq(uint32_t d_tmem, uint64_t a_kv, uint64_t b_q) {
  using Lay = BwdLayout<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false, false);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    const uint32_t off = (k >> 2) * Lay::kBox + (k & 3) * 32;
    umma_bf16_ss(d_tmem, sdesc_step(a_kv, off), sdesc_step(b_q, off), idesc, k > 0 ? 1u : 0u);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
               const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_k1,
               const __grid_constant__ CUtensorMap tm_v0, const __grid_constant__ CUtensorMap tm_v1,
               const __grid_constant__ CUtensorMap tm_do0,
               const __grid_constant__ CUtensorMap tm_do1,
               const __grid_constant__ CUtensorMap tm_lse,
               const __grid_constant__ CUtensorMap tm_dsum,
               const __grid_constant__ CUtensorMap tm_dqacc, const BwdParams p) {
  using Lay = BwdLayout<D>;
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {  // layout below needs a 1024-aligned window
    if (threadIdx.x == 0) atomicExch(p.status, DEV_MISALIGNED);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Lay::kBar);
  uint32_t* tmem_base_sh = reinterpret_cast<uint32_t*>(smem + Lay::kMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + Lay::kMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // CTA order.  kv_major: (batch, KV head) outer, task inner, so the CTAs
  // resident together hold key tiles of one KV head, walk the same query
  // tiles of the same few query heads and share those Q / dO tiles and dQ
  // rows in L2 (long sequences: many waves of similar-length tasks per KV
  // head).  Otherwise task outer: the heaviest tasks of every KV head run
  // together, so a wave holds tasks of similar length (short sequences).
  const int hb = p.Hkv * p.batch;
  const int n_tasks = static_cast<int>(gridDim.x) / hb;
  int task, rem;
  if (p.kv_major) {
    task = static_cast<int>(blockIdx.x) % n_tasks;
    rem = static_cast<int>(blockIdx.x) / n_tasks;
  } else {
    task = static_cast<int>(blockIdx.x) / hb;
    rem = static_cast<int>(blockIdx.x) - task * hb;
  }
  const int bz = rem / p.Hkv;
  const int kvh = rem - bz * p.Hkv;
  const int32_t* tw = p.tasks + static_cast<int64_t>(task) * kTaskWords;
  const int k_stream = tw[0];
  const int k_tile = tw[1];
  const int32_t* segs = p.segs + static_cast<int64_t>(tw[3]) * kSegWords;
  const int n_segs = tw[4];
  const int n_steps = tw[5] * p.G;
  const bool accumulate = (tw[6] & 1) != 0;  // dK/dV into the fp32 accumulators
#ifdef CSBP_DEBUG_CHECKS
  {
    bool bad = false;
    if (threadIdx.x == 0) {
      bad = !task_record_ok(tw, p.segs, p.n_segs, p.nT);
      if (bad) atomicExch(p.status, DEV_BADWORK);
    }
    if (__syncthreads_or(bad)) return;  // nothing issued yet
  }
#endif

  if (threadIdx.x == 0) {
    for (int i = 0; i < C_COUNT; ++i) {
      int count = 1;
      if (i == C_P_READY || i == C_DS_READY || i == C_DQ_FREE) count = 8;  // all compute warps
      if (i == C_STAGE_FULL || i == C_STAGE_FULL + 1) count = 4;            // warps of one half
      mbar_init(&bars[i], count);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (D == 64) {  // zero rows of K^T for the padded dQ^T MMA
    uint4* z = reinterpret_cast<uint4*>(smem + Lay::kZero);
    for (int i = threadIdx.x; i < Lay::kBox / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_base_sh;

  const uint32_t sK = smem_u32(smem + Lay::kK);
  const uint32_t sV = smem_u32(smem + Lay::kV);
  const uint32_t sQ = smem_u32(smem + Lay::kQ);
  const uint32_t sDO = smem_u32(smem + Lay::kDO);
  const uint32_t sX = smem_u32(smem + Lay::kX);

  if (n_steps > 0 && warp == 0 && lane == 0) {
    // ===================== TMA producer: K, V, then Q + LSE + D per step
    const void* tk = k_stream ? static_cast<const void*>(&tm_k1) : static_cast<const void*>(&tm_k0);
    const void* tv = k_stream ? static_cast<const void*>(&tm_v1) : static_cast<const void*>(&tm_v0);
    mbar_arrive_expect_tx(&bars[C_KV_FULL], 2 * Lay::kTileBytes);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(smem + Lay::kK + c * Lay::kBox, tk, &bars[C_KV_FULL], kvh * D + c * 64,
                  k_tile * kTile, bz);
      tma_load_3d(smem + Lay::kV + c * Lay::kBox, tv, &bars[C_KV_FULL], kvh * D + c * 64,
                  k_tile * kTile, bz);
    }
    QWalk w;
    w.start(segs, n_segs, p.G, p.window > 0);
    int nq = 0;
    bool ok = true;
    for (int i = 0; i < n_steps && ok; ++i, w.next()) {
      const int h = kvh * p.G + w.g;
      const int qs = w.stream;
      const int q0 = w.t * kTile;
      const void* tq = qs ? static_cast<const void*>(&tm_q1) : static_cast<const void*>(&tm_q0);
      const int st = i % kStages;
      if (i >= kStages)
        ok = mbar_wait(&bars[C_Q_EMPTY + st], ((i / kStages) - 1) & 1, p.status, abort_flag);
      if (!ok) break;
      mbar_arrive_expect_tx(&bars[C_Q_FULL + st], Lay::kTileBytes + Lay::kStatBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + Lay::kQ + st * Lay::kTileBytes + c * Lay::kBox, tq, &bars[C_Q_FULL + st],
                    h * D + c * 64, q0, bz);
      uint8_t* stat = smem + Lay::kStat + st * Lay::kStatBytes;
      tma_load_2d(stat, &tm_lse, &bars[C_Q_FULL + st], q0, (bz * 2 + qs) * p.Hq + h);
      tma_load_2d(stat + kTile * 4, &tm_dsum, &bars[C_Q_FULL + st], q0,
                  (qs * p.batch + bz) * p.Hq + h);
      nq = i + 1;
    }
    if (!ok) {
      mbar_wait(&bars[C_KV_FULL], 0, nullptr, nullptr, 200000000ull);
      for (int i = (nq > kStages ? nq - kStages : 0); i < nq; ++i)
        mbar_wait(&bars[C_Q_FULL + i % kStages], (i / kStages) & 1, nullptr, nullptr, 200000000ull);
    }
  } else if (n_steps > 0 && warp == 2 && lane == 0) {
    // ===================== TMA producer: dO per step
    QWalk w;
    w.start(segs, n_segs, p.G, p.window > 0);
    int ndo = 0;
    bool ok = true;
    for (int i = 0; i < n_steps && ok; ++i, w.next()) {
      const int h = kvh * p.G + w.g;
      const void* td = w.stream ? static_cast<const void*>(&tm_do1) : static_cast<const void*>(&tm_do0);
      const int st = i % Lay::kDOStages;
      if (i >= Lay::kDOStages)
        ok = mbar_wait(&bars[C_DO_EMPTY + st], ((i / Lay::kDOStages) - 1) & 1, p.status, abort_flag);
      if (!ok) break;
      mbar_arrive_expect_tx(&bars[C_DO_FULL + st], Lay::kTileBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + Lay::kDO + st * Lay::kTileBytes + c * Lay::kBox, td,
                    &bars[C_DO_FULL + st], h * D + c * 64, w.t * kTile, bz);
      ndo = i + 1;
    }
    if (!ok) {
      for (int i = (ndo > Lay::kDOStages ? ndo - Lay::kDOStages : 0); i < ndo; ++i)
        mbar_wait(&bars[C_DO_FULL + i % Lay::kDOStages], (i / Lay::kDOStages) & 1, nullptr, nullptr,
                  200000000ull);
    }
  } else if (n_steps > 0 && warp == 1 && lane == 0) {
    // ===================== MMA issuer
    constexpr uint32_t idesc_kd = idesc_bf16_f32(128, D, false, true);   // dV, dK
    constexpr uint32_t idesc_q = idesc_bf16_f32(128, 128, true, true);   // dQ^T
    auto wait_q = [&](int i) {
      return mbar_wait_spin(&bars[C_Q_FULL + i % kStages], (i / kStages) & 1, p.status, abort_flag);
    };
    auto wait_do = [&](int i) {
      return mbar_wait_spin(&bars[C_DO_FULL + i % Lay::kDOStages], (i / Lay::kDOStages) & 1, p.status,
                       abort_flag);
    };
    const uint64_t k_kmaj = sdesc_sw128(sK, 16, 1024);   // K as K-major A (S^T)
    const uint64_t v_kmaj = sdesc_sw128(sV, 16, 1024);   // V as K-major A (dP^T)
    const uint64_t k_mn = sdesc_sw128(                   // K^T as MN-major A (dQ^T)
        sK, (D == 64) ? static_cast<uint32_t>(Lay::kZero - Lay::kK) : Lay::kBox, 1024);
    const uint64_t x_kmaj = sdesc_sw128(sX, 16, 1024);           // dS^T as K-major A (dK)
    const uint64_t x_mn = sdesc_sw128(sX, Lay::kXBox, 1024);     // dS^T as MN-major B (dQ^T)
    bool ok = mbar_wait_spin(&bars[C_KV_FULL], 0, p.status, abort_flag) && wait_q(0) && wait_do(0);
    if (ok) {
      tc_fence_after_sync();
      issue_kq<D>(tmem + Lay::kColS, k_kmaj, sdesc_sw128(sQ, 16, 1024));
      umma_commit(&bars[C_S_FULL]);
      issue_kq<D>(tmem + Lay::kColDP, v_kmaj, sdesc_sw128(sDO, 16, 1024));
      umma_commit(&bars[C_DP_FULL]);
    }
    for (int i = 0; i < n_steps && ok; ++i) {
      const int st = i % kStages;
      const uint32_t q_s = sQ + st * Lay::kTileBytes;
      const uint32_t do_s = sDO + (i % Lay::kDOStages) * Lay::kTileBytes;
      const uint32_t acc0 = i > 0 ? 1u : 0u;
      // ---- dV += P^T dO, P^T in TMEM: half h's 32 packed columns at 64h
      if (!mbar_wait_spin(&bars[C_P_READY], i & 1, p.status, abort_flag)) break;
      tc_fence_after_sync();
      {
        const uint64_t b = sdesc_sw128(do_s, Lay::kBox, 1024);  // dO as MN-major B
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_bf16_ts(tmem + Lay::kColDV, tmem + Lay::kColS + (kk >> 2) * kHalf + (kk & 3) * 8,
                       sdesc_step(b, kk * 2048), idesc_kd, kk > 0 ? 1u : acc0);
      }
      umma_commit(&bars[C_PV_DONE]);
      umma_commit(&bars[C_DO_EMPTY + i % Lay::kDOStages]);
      // ---- dQ^T = K^T dS^T first (the compute warps wait on it), then
      //      dK += dS^T Q
      if (!mbar_wait_spin(&bars[C_DS_READY], i & 1, p.status, abort_flag)) break;
      tc_fence_after_sync();
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        umma_bf16_ss(tmem + Lay::kColDP, sdesc_step(k_mn, kk * 2048), sdesc_step(x_mn, kk * 2048),
                     idesc_q, kk > 0 ? 1u : 0u);
      umma_commit(&bars[C_DQ_FULL]);
      {
        const uint64_t b = sdesc_sw128(q_s, Lay::kBox, 1024);  // Q as MN-major B
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_bf16_ss(tmem + Lay::kColDK, sdesc_step(x_kmaj, (kk >> 2) * Lay::kXBox + (kk & 3) * 32),
                       sdesc_step(b, kk * 2048), idesc_kd, kk > 0 ? 1u : acc0);
      }
      umma_commit(&bars[C_DK_DONE]);
      umma_commit(&bars[C_Q_EMPTY + st]);
      if (i + 1 < n_steps) {
        // ---- S^T_{i+1}: its columns held P^T_i, consumed once dV_i is done
        if (!mbar_wait_spin(&bars[C_PV_DONE], i & 1, p.status, abort_flag) || !wait_q(i + 1)) break;
        tc_fence_after_sync();
        issue_kq<D>(tmem + Lay::kColS, k_kmaj,
                    sdesc_sw128(sQ + ((i + 1) % kStages) * Lay::kTileBytes, 16, 1024));
        umma_commit(&bars[C_S_FULL]);
        // ---- dP^T_{i+1}: its columns held dQ^T_i, free once both halves copied it
        if (!mbar_wait_spin(&bars[C_DQ_FREE], i & 1, p.status, abort_flag) || !wait_do(i + 1)) break;
        tc_fence_after_sync();
        issue_kq<D>(tmem + Lay::kColDP, v_kmaj,
                    sdesc_sw128(sDO + ((i + 1) % Lay::kDOStages) * Lay::kTileBytes, 16, 1024));
        umma_commit(&bars[C_DP_FULL]);
      }
    }
    umma_commit(&bars[C_ACC_DONE]);
    umma_commit(&bars[C_DRAIN]);
    mbar_wait(&bars[C_DRAIN], 0, nullptr, nullptr, 500000000ull);
  } else if (warp >= 4) {
    // ===================== compute halves
    const int hf = (warp >= 8) ? 1 : 0;          // query-column half of this warpgroup
    const int r = (warp & 3) * 32 + lane;         // key row (TMEM lane)
    const bool leader = (warp & 3) == 0;          // issues this half's dQ reduce-adds
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t colS = Lay::kColS + hf * kHalf;
    const uint32_t colDP = Lay::kColDP + hf * kHalf;
    const int kpos = k_tile * kTile + r;
    const bool k_valid = kpos < p.L;
    const int kb = k_valid ? kpos / p.M : -1;
    const float sl2 = p.scale_log2;
    uint8_t* xbox = smem + Lay::kX + hf * Lay::kXBox;
    // dQ rows [0, kRowsX) of the half are staged in its dS^T box, the rest in
    // its own buffer, both as [row][d] fp32
    float* stage_x = reinterpret_cast<float*>(xbox);
    float* stage_sq = reinterpret_cast<float*>(smem + Lay::kSQ) + hf * Lay::kRowsSQ * D;
    const bool k_ragged = (k_tile + 1) * kTile > p.L;
    QWalk wk;
    wk.start(segs, n_segs, p.G, p.window > 0);
    bool ok = true;
    for (int i = 0; i < n_steps; ++i, wk.next()) {
      const int qs = wk.stream;
      const int h = kvh * p.G + wk.g;
      const int q0 = wk.t * kTile + hf * kHalf;   // first query row of this half
      const int st = i % kStages;
      if (!mbar_wait_warp(&bars[C_S_FULL], i & 1, p.status, abort_flag) ||
          !mbar_wait_warp(&bars[C_Q_FULL + st], (i / kStages) & 1, p.status, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float* lse =
          reinterpret_cast<const float*>(smem + Lay::kStat + st * Lay::kStatBytes) + hf * kHalf;
      const float* Dq = lse + kTile;
      const float2* lse2 = reinterpret_cast<const float2*>(lse);
      const float2* Dq2 = reinterpret_cast<const float2*>(Dq);
      const uint64_t sl2x2 = f2_pack(sl2, sl2);
      const bool masked = (wk.flags & 1) || k_ragged || (q0 + kHalf > p.L);
      // ---- P^T = exp(S^T scale - LSE), written back to TMEM as bf16 pairs
      float pr[kHalf];
      tmem_ld32x2(tmem + lane_base + colS, tmem + lane_base + colS + 32, pr, pr + 32);
      if (masked) {
        // allowed query positions of this key row form one range [lo, hi);
        // 32 columns that no key row of the warp may read give P^T = 0
        // without their exponentials (the special-function unit bounds this)
        int lo, hi;
        allowed_query_range(qs, k_stream, kpos, kb, p.M, p.L, p.window, p.clean_causal, k_valid,
                            lo, hi);
        lo -= q0;
        hi -= q0;
#pragma unroll
        for (int q = 0; q < kHalf / 32; ++q) {
          const int c0 = q * 32;
          if (__all_sync(0xffffffffu, hi <= c0 || lo >= c0 + 32)) {
#pragma unroll
            for (int c = c0; c < c0 + 32; ++c) pr[c] = 0.f;
          } else {
#pragma unroll
            for (int c = c0; c < c0 + 32; c += 2) {
              float e0, e1;
              p_exp2(pr[c], pr[c + 1], lse2[c / 2], sl2x2, e0, e1);
              pr[c] = (c >= lo && c < hi) ? e0 : 0.f;
              pr[c + 1] = (c + 1 >= lo && c + 1 < hi) ? e1 : 0.f;
            }
          }
        }
      } else {
#pragma unroll
        for (int c = 0; c < kHalf; c += 2) p_exp2(pr[c], pr[c + 1], lse2[c / 2], sl2x2, pr[c], pr[c + 1]);
      }
      {
        float packed[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) packed[c] = __uint_as_float(pack_bf16x2(pr[2 * c], pr[2 * c + 1]));
        tmem_st32(tmem + lane_base + colS, packed);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_P_READY]);
      // ---- dS^T = P^T o (dP^T - D) into this half's box, once the reduce-add
      //      of the dQ rows staged there in the previous step has read them
      //      (it was left in flight over the P^T work; the one of the own
      //      buffer, issued after it, may still be)
      if (i > 0 && leader && lane == 0) {
        if (Lay::kRowsSQ > 0)
          bulk_wait_group_read<1>();
        else
          bulk_wait_group_read<0>();
        mbar_arrive(&bars[C_X_FREE + hf]);
      }
      if (!mbar_wait_warp(&bars[C_DP_FULL], i & 1, p.status, abort_flag) ||
          (i > 0 && !mbar_wait_warp(&bars[C_X_FREE + hf], (i - 1) & 1, p.status, abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      {
        float a[32], b[32];
        tmem_ld32x2(tmem + lane_base + colDP, tmem + lane_base + colDP + 32, a, b);
#pragma unroll
        for (int chunk = 0; chunk < kHalf / 8; ++chunk) {
          const float* dp = (chunk < 4) ? a + chunk * 8 : b + (chunk - 4) * 8;
          const int c0 = chunk * 8;
          uint4 v;
          v.x = ds_pair(pr[c0 + 0], pr[c0 + 1], dp[0], dp[1], Dq2[c0 / 2 + 0]);
          v.y = ds_pair(pr[c0 + 2], pr[c0 + 3], dp[2], dp[3], Dq2[c0 / 2 + 1]);
          v.z = ds_pair(pr[c0 + 4], pr[c0 + 5], dp[4], dp[5], Dq2[c0 / 2 + 2]);
          v.w = ds_pair(pr[c0 + 6], pr[c0 + 7], dp[6], dp[7], Dq2[c0 / 2 + 3]);
          *reinterpret_cast<uint4*>(xbox + sw128_offset(r, chunk)) = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_DS_READY]);
      // ---- dQ^T: thread r owns head-dim row r of this half's 64 query columns
      if (!mbar_wait_warp(&bars[C_DQ_FULL], i & 1, p.status, abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      float dq[kHalf];
      tmem_ld32x2(tmem + lane_base + colDP, tmem + lane_base + colDP + 32, dq, dq + 32);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_DQ_FREE]);
      // stage the half's 64 dQ rows: the last kRowsSQ in its own buffer once
      // the previous step's reduce-add from there has read it, the first
      // kRowsX in its dS^T box once dK_i (the box's last reader) is done
      if (Lay::kRowsSQ > 0) {
        if (i > 0 && leader && lane == 0) {
          bulk_wait_group_read<0>();
          mbar_arrive(&bars[C_SQ_FREE + hf]);
        }
        if (i > 0 && !mbar_wait_warp(&bars[C_SQ_FREE + hf], (i - 1) & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        if (r < D) {
#pragma unroll
          for (int c = 0; c < Lay::kRowsSQ; ++c) stage_sq[c * D + r] = dq[Lay::kRowsX + c];
        }
      }
      if (!mbar_wait_warp(&bars[C_DK_DONE], i & 1, p.status, abort_flag)) {
        ok = false;
        break;
      }
      if (r < D) {
#pragma unroll
        for (int c = 0; c < Lay::kRowsX; ++c) stage_x[c * D + r] = dq[c];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_STAGE_FULL + hf]);
      if (leader) {
        if (!mbar_wait_warp(&bars[C_STAGE_FULL + hf], i & 1, p.status, abort_flag)) {
          ok = false;
          break;
        }
        // one bulk group per buffer, the dS^T box first (its rows are needed
        // back soonest); rows past L (ragged last tile) are dropped, leaving
        // an empty group
        if (lane == 0) {
          const int plane = qs * p.batch + bz;
          if (q0 < p.L) tma_reduce_add_3d(&tm_dqacc, stage_x, h * D, q0, plane);
          bulk_commit_group();
          if (Lay::kRowsSQ > 0) {
            if (q0 + Lay::kRowsX < p.L)
              tma_reduce_add_3d(&tm_dqacc, stage_sq, h * D, q0 + Lay::kRowsX, plane);
            bulk_commit_group();
          }
        }
        __syncwarp();
      }
    }
    if (leader && lane == 0) bulk_wait_group<0>();  // reduce-adds complete before exit
    // ---- epilogue (half 0): dV, dK rows of this key tile
    if (hf == 0) {
      __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(k_stream ? p.dv[1] : p.dv[0]) +
                          ((static_cast<int64_t>(bz) * p.L + kpos) * p.Hkv + kvh) * D;
      __nv_bfloat16* dk = static_cast<__nv_bfloat16*>(k_stream ? p.dk[1] : p.dk[0]) +
                          ((static_cast<int64_t>(bz) * p.L + kpos) * p.Hkv + kvh) * D;
      if (n_steps == 0) {
        if (k_valid && !accumulate) {
          for (int c = 0; c < D; c += 8) {
            *reinterpret_cast<uint4*>(dv + c) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(dk + c) = make_uint4(0, 0, 0, 0);
          }
        }
      } else if (ok && mbar_wait_warp(&bars[C_ACC_DONE], 0, p.status, abort_flag)) {
        tc_fence_after_sync();
        // windowed tasks add their share into the fp32 accumulators
        const int64_t acc_row =
            ((static_cast<int64_t>(k_stream) * p.batch + bz) * p.L + kpos) * p.Hkv + kvh;
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          __nv_bfloat16* dstp = half ? dk : dv;
          const uint32_t col = half ? Lay::kColDK : Lay::kColDV;
          const float mul = half ? p.scale : 1.f;
          float* accp = (half ? p.dk_acc : p.dv_acc);
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            float v[32];
            tmem_ld32(tmem + lane_base + col + ch * 32, v);
            if (k_valid && accumulate) {
              float4* a4 = reinterpret_cast<float4*>(accp + acc_row * D + ch * 32);
#pragma unroll
              for (int e = 0; e < 8; ++e)
                atomicAdd(a4 + e, make_float4(v[4 * e] * mul, v[4 * e + 1] * mul, v[4 * e + 2] * mul,
                                              v[4 * e + 3] * mul));
            } else if (k_valid) {
#pragma unroll
              for (int e = 0; e < 32; e += 8) {
                uint4 u;
                u.x = pack_bf16x2(v[e] * mul, v[e + 1] * mul);
                u.y = pack_bf16x2(v[e + 2] * mul, v[e + 3] * mul);
                u.z = pack_bf16x2(v[e + 4] * mul, v[e + 5] * mul);
                u.w = pack_bf16x2(v[e + 6] * mul, v[e + 7] * mul);
                *reinterpret_cast<uint4*>(dstp + ch * 32 + e) = u;
              }
            }
          }
        }
      }
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

}  // namespace

template <int D>
static cudaError_t launch_bwd_d(const CUtensorMap* maps, const BwdParams& p, int n_tasks,
                                cudaStream_t stream) {
  using Lay = BwdLayout<D>;
  // the shared-memory limit is a per-device attribute: set it once on each
  static PerDeviceOnce configured;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!configured.run(dev, [&](int) {
        e = cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 Lay::kDynSmem);
        return e == cudaSuccess;
      }))
    return e != cudaSuccess ? e : cudaErrorInvalidDevice;
  const int64_t grid = static_cast<int64_t>(n_tasks) * p.Hkv * p.batch;
  if (grid <= 0) return cudaSuccess;
  bwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, Lay::kDynSmem, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], maps[8], maps[9],
      maps[10], p);
  return cudaGetLastError();
}

// Rows of one TMA box for the query-side maps (Q, dO) and the LSE/D maps.
int bwd_query_box_rows() { return kTile; }
// Query rows of one dQ reduce-add box: a 16 KB fp32 box of d columns.
int bwd_dq_box_rows(int d) { return (kTile * kHalf * 2) / (d * 4); }

// maps: q_clean, q_corr, k_clean, k_corr, v_clean, v_corr, do_clean, do_corr
//       (128-row boxes), lse ({L, batch*2*Hq} fp32) and dsum ({L, 2*batch*Hq}
//       fp32) with 128-position boxes, dq_acc ({Hq*d, L, 2*batch} fp32, box
//       {d, 32, 1}, no swizzle)
cudaError_t launch_bwd(int d, const CUtensorMap* maps, const BwdParams& p, int n_tasks,
                       cudaStream_t stream) {
  if (d == 128) return launch_bwd_d<128>(maps, p, n_tasks, stream);
  return launch_bwd_d<64>(maps, p, n_tasks, stream);
}

}  // namespace csbp
