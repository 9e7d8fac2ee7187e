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
// query tile is processed as two 64-row sub-tiles by two compute warpgroups
// that alternate, so the tensor core works on one sub-tile while the other
// warpgroup computes exponentials.  Roles (384 threads):
//   warp 0 lane 0  TMA producer: K, V once; per sub-tile Q (3 stages) with its
//                  LSE and D slices, and dO (2 stages)
//   warp 1 lane 0  MMA issuer, per sub-tile s (stream w = s & 1):
//                    dV += P_s^T dO_s   (P^T read from TMEM)
//                    dK += dS_s^T Q_s;  dQ_s^T = K^T dS_s^T  (dS^T from smem)
//                    then dP^T_{s+1} = V dO_{s+1}^T and S^T_{s+2} = K Q_{s+2}^T
//   warps 4..7 / 8..11  compute streams 0 / 1: thread t owns key row t (TMEM
//                  lane t).  It turns S^T into P^T (bf16, written back over
//                  its own S^T columns of TMEM) and dP^T into dS^T (bf16,
//                  into the stream's 128B-swizzled shared tile: the K-major A
//                  operand of dK and the MN-major B operand of dQ^T).  Then it
//                  copies dQ^T (thread t = head-dim row t) out of TMEM into a
//                  shared staging tile, from which one TMA bulk reduce-add per
//                  32 query rows adds it into the fp32 dQ accumulator.
// TMEM columns: stream w has S^T (then P^T) at 128w and dP^T (then dQ^T) at
// 128w + 64; dV at 256, dK at 256 + d.  For d = 64 the dQ^T MMA runs with
// M = 128 and the upper 64 rows of K^T read a zero tile.
#include <cuda.h>
#include <cuda_runtime.h>

#include "csbp_internal.h"
#include "ptx_sm100.cuh"

namespace csbp {

namespace {

constexpr int kThreads = 384;
constexpr int kSub = 64;          // query rows per sub-tile
constexpr int kQStages = 3;
constexpr int kDOStages = 2;
constexpr int kStageRows = 32;    // query rows per dQ reduce-add
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdLayout {
  static constexpr int kKVBytes = kTile * D * 2;     // K or V tile
  static constexpr int kKVBox = kTile * 128;         // one 64-column box of K/V
  static constexpr int kSubBytes = kSub * D * 2;     // Q or dO sub-tile
  static constexpr int kSubBox = kSub * 128;         // one 64-column box of a sub-tile
  static constexpr int kXBytes = kTile * kSub * 2;   // dS^T of one stream
  static constexpr int kStageBytes = kStageRows * D * 4;  // fp32 dQ rows of one stream
  static constexpr int kStatBytes = 2 * kSub * 4;    // LSE and D of one sub-tile
  static constexpr int kK = 0;
  static constexpr int kV = kK + kKVBytes;
  static constexpr int kZero = kV + kKVBytes;        // zero K^T rows (d = 64 only)
  static constexpr int kQ = kZero + (D == 64 ? kKVBox : 0);
  static constexpr int kDO = kQ + kQStages * kSubBytes;
  static constexpr int kX = kDO + kDOStages * kSubBytes;
  static constexpr int kStage = kX + 2 * kXBytes;
  static constexpr int kStat = kStage + 2 * kStageBytes;
  static constexpr int kBytes = kStat + kQStages * kStatBytes;
  static constexpr int kDynSmem = kBytes + 1024;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + D;
};

enum BwdBar {
  C_KV_FULL = 0,
  C_Q_FULL,                          // [kQStages]
  C_Q_EMPTY = C_Q_FULL + kQStages,   // [kQStages]
  C_DO_FULL = C_Q_EMPTY + kQStages,  // [kDOStages]
  C_DO_EMPTY = C_DO_FULL + kDOStages,
  C_S_FULL = C_DO_EMPTY + kDOStages,  // per stream [2] from here on
  C_DP_FULL = C_S_FULL + 2,
  C_P_READY = C_DP_FULL + 2,
  C_PV_DONE = C_P_READY + 2,
  C_DS_READY = C_PV_DONE + 2,
  C_X_FREE = C_DS_READY + 2,
  C_DQ_FULL = C_X_FREE + 2,
  C_DQ_FREE = C_DQ_FULL + 2,
  C_STAGE_FULL = C_DQ_FREE + 2,
  C_STAGE_FREE = C_STAGE_FULL + 2,
  C_ACC_DONE = C_STAGE_FREE + 2,
  C_DRAIN,
  C_COUNT
};

// Walk over (query head in group, segment, 128-row query tile) of a task.
struct QWalk {
  const int32_t* seg0;
  int n_segs, g, si, t, end, stream, flags;
  __device__ void load_seg() {
    const int32_t* s = seg0 + si * kSegWords;
    stream = s[0];
    t = s[1];
    end = s[2];
    flags = s[3];
  }
  __device__ void start(const int32_t* s, int n) {
    seg0 = s;
    n_segs = n;
    g = 0;
    si = 0;
    if (n > 0) load_seg();
  }
  __device__ void next() {
    if (++t < end) return;
    if (++si >= n_segs) {
      si = 0;
      ++g;
    }
    load_seg();
  }
};

// Query positions [lo, hi) that may read key block kb of copy k_stream, for
// queries of copy q_stream: clean keys are read by clean queries of the same
// or later blocks and by corrupted queries of later blocks; corrupted keys
// only by corrupted queries of their own block.
__device__ __forceinline__ void allowed_query_range(int q_stream, int k_stream, int kb, int M,
                                                    int L, bool k_valid, int& lo, int& hi) {
  if (!k_valid || (q_stream == 0 && k_stream == 1)) {
    lo = hi = 0;
    return;
  }
  if (k_stream == 0) {
    lo = (q_stream == 0) ? kb * M : (kb + 1) * M;
    hi = L;
  } else {
    lo = kb * M;
    hi = min((kb + 1) * M, L);
  }
}

// S^T (or dP^T) of one sub-tile: M = 128 key rows, N = 64 query rows, K = d.
// a_kv / b_sub: K-major base descriptors of the key-side tile and the
// query-side sub-tile.
template <int D>
__device__ __forceinline__ void issue_kq(uint32_t d_tmem, uint64_t a_kv, uint64_t b_sub) {
  using Lay = BwdLayout<D>;
  constexpr uint32_t idesc = idesc_bf16_f32(128, kSub, false, false);
#pragma unroll
  for (int k = 0; k < D / 16; ++k) {
    umma_bf16_ss(d_tmem, sdesc_step(a_kv, (k >> 2) * Lay::kKVBox + (k & 3) * 32),
                 sdesc_step(b_sub, (k >> 2) * Lay::kSubBox + (k & 3) * 32), idesc, k > 0 ? 1u : 0u);
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
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[C_COUNT];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int hb = p.Hkv * p.batch;
  const int task = blockIdx.x / hb;
  const int rem = blockIdx.x - task * hb;
  const int bz = rem / p.Hkv;
  const int kvh = rem - bz * p.Hkv;
  const int32_t* tw = p.tasks + static_cast<int64_t>(task) * kTaskWords;
  const int k_stream = tw[0];
  const int k_tile = tw[1];
  const int32_t* segs = p.segs + static_cast<int64_t>(tw[3]) * kSegWords;
  const int n_segs = tw[4];
  const int n_sub = 2 * tw[5] * p.G;  // two 64-row sub-tiles per query tile

  if (threadIdx.x == 0) {
    for (int i = 0; i < C_COUNT; ++i) {
      const bool per_warp = (i >= C_P_READY && i < C_P_READY + 2) ||
                            (i >= C_DS_READY && i < C_DS_READY + 2) ||
                            (i >= C_DQ_FREE && i < C_DQ_FREE + 2) ||
                            (i >= C_STAGE_FULL && i < C_STAGE_FULL + 2);
      mbar_init(&bars[i], per_warp ? 4 : 1);
    }
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (D == 64) {  // zero rows of K^T for the padded dQ^T MMA
    uint4* z = reinterpret_cast<uint4*>(smem + Lay::kZero);
    for (int i = threadIdx.x; i < Lay::kKVBox / 16; i += kThreads) z[i] = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  const uint32_t sK = smem_u32(smem + Lay::kK);
  const uint32_t sV = smem_u32(smem + Lay::kV);
  const uint32_t sQ = smem_u32(smem + Lay::kQ);
  const uint32_t sDO = smem_u32(smem + Lay::kDO);
  const uint32_t sX = smem_u32(smem + Lay::kX);

  if (n_sub > 0 && warp == 0 && lane == 0) {
    // ===================== TMA producer
    const void* tk = k_stream ? static_cast<const void*>(&tm_k1) : static_cast<const void*>(&tm_k0);
    const void* tv = k_stream ? static_cast<const void*>(&tm_v1) : static_cast<const void*>(&tm_v0);
    mbar_arrive_expect_tx(&bars[C_KV_FULL], 2 * Lay::kKVBytes);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(smem + Lay::kK + c * Lay::kKVBox, tk, &bars[C_KV_FULL], kvh * D + c * 64,
                  k_tile * kTile, bz);
      tma_load_3d(smem + Lay::kV + c * Lay::kKVBox, tv, &bars[C_KV_FULL], kvh * D + c * 64,
                  k_tile * kTile, bz);
    }
    QWalk w;
    w.start(segs, n_segs);
    int nq = 0, ndo = 0;
    bool ok = true;
    for (int s = 0; s < n_sub && ok; ++s) {
      const int h = kvh * p.G + w.g;
      const int qs = w.stream;
      const int q0 = w.t * kTile + (s & 1) * kSub;
      const void* tq = qs ? static_cast<const void*>(&tm_q1) : static_cast<const void*>(&tm_q0);
      const void* td = qs ? static_cast<const void*>(&tm_do1) : static_cast<const void*>(&tm_do0);
      const int qst = s % kQStages;
      if (s >= kQStages)
        ok = mbar_wait(&bars[C_Q_EMPTY + qst], ((s / kQStages) - 1) & 1, p.status, &abort_flag);
      if (!ok) break;
      mbar_arrive_expect_tx(&bars[C_Q_FULL + qst], Lay::kSubBytes + Lay::kStatBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + Lay::kQ + qst * Lay::kSubBytes + c * Lay::kSubBox, tq,
                    &bars[C_Q_FULL + qst], h * D + c * 64, q0, bz);
      uint8_t* stat = smem + Lay::kStat + qst * Lay::kStatBytes;
      tma_load_2d(stat, &tm_lse, &bars[C_Q_FULL + qst], q0, (bz * 2 + qs) * p.Hq + h);
      tma_load_2d(stat + kSub * 4, &tm_dsum, &bars[C_Q_FULL + qst], q0,
                  (qs * p.batch + bz) * p.Hq + h);
      nq = s + 1;
      const int dst = s % kDOStages;
      if (s >= kDOStages)
        ok = mbar_wait(&bars[C_DO_EMPTY + dst], ((s / kDOStages) - 1) & 1, p.status, &abort_flag);
      if (!ok) break;
      mbar_arrive_expect_tx(&bars[C_DO_FULL + dst], Lay::kSubBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + Lay::kDO + dst * Lay::kSubBytes + c * Lay::kSubBox, td,
                    &bars[C_DO_FULL + dst], h * D + c * 64, q0, bz);
      ndo = s + 1;
      if (s & 1) w.next();
    }
    if (!ok) {
      // drain the loads that may still be in flight
      mbar_wait(&bars[C_KV_FULL], 0, nullptr, nullptr, 200000000ull);
      for (int s = (nq > kQStages ? nq - kQStages : 0); s < nq; ++s)
        mbar_wait(&bars[C_Q_FULL + s % kQStages], (s / kQStages) & 1, nullptr, nullptr, 200000000ull);
      for (int s = (ndo > kDOStages ? ndo - kDOStages : 0); s < ndo; ++s)
        mbar_wait(&bars[C_DO_FULL + s % kDOStages], (s / kDOStages) & 1, nullptr, nullptr,
                  200000000ull);
    }
  } else if (n_sub > 0 && warp == 1 && lane == 0) {
    // ===================== MMA issuer
    constexpr uint32_t idesc_kd = idesc_bf16_f32(128, D, false, true);  // dV, dK
    constexpr uint32_t idesc_q = idesc_bf16_f32(128, kSub, true, true);  // dQ^T
    auto qbuf = [&](int s) { return sQ + (s % kQStages) * Lay::kSubBytes; };
    auto dobuf = [&](int s) { return sDO + (s % kDOStages) * Lay::kSubBytes; };
    auto wait_q = [&](int s) {
      return mbar_wait(&bars[C_Q_FULL + s % kQStages], (s / kQStages) & 1, p.status, &abort_flag);
    };
    auto wait_do = [&](int s) {
      return mbar_wait(&bars[C_DO_FULL + s % kDOStages], (s / kDOStages) & 1, p.status, &abort_flag);
    };
    // base descriptors of the CTA-resident key-side tiles
    const uint64_t k_kmaj = sdesc_sw128(sK, 16, 1024);   // K as K-major A (S^T)
    const uint64_t v_kmaj = sdesc_sw128(sV, 16, 1024);   // V as K-major A (dP^T)
    const uint64_t k_mn = sdesc_sw128(                   // K^T as MN-major A (dQ^T)
        sK, (D == 64) ? static_cast<uint32_t>(Lay::kZero - Lay::kK) : Lay::kKVBox, 1024);
    bool ok = mbar_wait(&bars[C_KV_FULL], 0, p.status, &abort_flag) && wait_q(0) && wait_do(0);
    if (ok) {
      tc_fence_after_sync();
      issue_kq<D>(tmem + 0, k_kmaj, sdesc_sw128(qbuf(0), 16, 1024));
      umma_commit(&bars[C_S_FULL + 0]);
      issue_kq<D>(tmem + 64, v_kmaj, sdesc_sw128(dobuf(0), 16, 1024));
      umma_commit(&bars[C_DP_FULL + 0]);
      if (n_sub > 1) {
        ok = wait_q(1);
        if (ok) {
          tc_fence_after_sync();
          issue_kq<D>(tmem + 128, k_kmaj, sdesc_sw128(qbuf(1), 16, 1024));
          umma_commit(&bars[C_S_FULL + 1]);
        }
      }
    }
    for (int s = 0; s < n_sub && ok; ++s) {
      const int w = s & 1;
      const int k = s >> 1;
      const uint32_t xw = sX + w * Lay::kXBytes;
      const uint32_t acc0 = s > 0 ? 1u : 0u;  // dV / dK accumulate after the first sub-tile
      // ---- dV += P^T dO (P^T in TMEM over the stream's S^T columns)
      if (!mbar_wait(&bars[C_P_READY + w], k & 1, p.status, &abort_flag)) break;
      tc_fence_after_sync();
      {
        const uint64_t b = sdesc_sw128(dobuf(s), Lay::kSubBox, 1024);  // dO as MN-major B
#pragma unroll
        for (int kk = 0; kk < kSub / 16; ++kk)
          umma_bf16_ts(tmem + Lay::kColDV, tmem + w * 128 + kk * 8, sdesc_step(b, kk * 2048),
                       idesc_kd, kk > 0 ? 1u : acc0);
      }
      umma_commit(&bars[C_PV_DONE + w]);
      umma_commit(&bars[C_DO_EMPTY + s % kDOStages]);
      // ---- dK += dS^T Q; dQ^T = K^T dS^T
      if (!mbar_wait(&bars[C_DS_READY + w], k & 1, p.status, &abort_flag)) break;
      tc_fence_after_sync();
      {
        const uint64_t a = sdesc_sw128(xw, 16, 1024);                  // dS^T as K-major A
        const uint64_t b = sdesc_sw128(qbuf(s), Lay::kSubBox, 1024);   // Q as MN-major B
#pragma unroll
        for (int kk = 0; kk < kSub / 16; ++kk)
          umma_bf16_ss(tmem + Lay::kColDK, sdesc_step(a, kk * 32), sdesc_step(b, kk * 2048), idesc_kd,
                       kk > 0 ? 1u : acc0);
        const uint64_t bx = sdesc_sw128(xw, Lay::kXBytes, 1024);        // dS^T as MN-major B
#pragma unroll
        for (int kk = 0; kk < kTile / 16; ++kk)
          umma_bf16_ss(tmem + w * 128 + 64, sdesc_step(k_mn, kk * 2048), sdesc_step(bx, kk * 2048),
                       idesc_q, kk > 0 ? 1u : 0u);
      }
      umma_commit(&bars[C_DQ_FULL + w]);
      umma_commit(&bars[C_Q_EMPTY + s % kQStages]);
      umma_commit(&bars[C_X_FREE + w]);
      // ---- dP^T of sub-tile s+1 (other stream; its columns held dQ^T_{s-1})
      if (s + 1 < n_sub) {
        const int w1 = w ^ 1;
        if ((s >= 1 && !mbar_wait(&bars[C_DQ_FREE + w1], ((s - 1) >> 1) & 1, p.status, &abort_flag)) ||
            !wait_do(s + 1))
          break;
        tc_fence_after_sync();
        issue_kq<D>(tmem + w1 * 128 + 64, v_kmaj, sdesc_sw128(dobuf(s + 1), 16, 1024));
        umma_commit(&bars[C_DP_FULL + w1]);
      }
      // ---- S^T of sub-tile s+2 (this stream): its columns held P^T_s, which
      //      dV_s has finished reading once PV_DONE completes
      if (s + 2 < n_sub) {
        if (!wait_q(s + 2) || !mbar_wait(&bars[C_PV_DONE + w], k & 1, p.status, &abort_flag)) break;
        tc_fence_after_sync();
        issue_kq<D>(tmem + w * 128, k_kmaj, sdesc_sw128(qbuf(s + 2), 16, 1024));
        umma_commit(&bars[C_S_FULL + w]);
      }
    }
    umma_commit(&bars[C_ACC_DONE]);
    umma_commit(&bars[C_DRAIN]);
    mbar_wait(&bars[C_DRAIN], 0, nullptr, nullptr, 500000000ull);
  } else if (warp >= 4) {
    // ===================== compute streams
    const int w = (warp >= 8) ? 1 : 0;
    const int r = threadIdx.x - 128 * (w + 1);  // key row (TMEM lane)
    const bool leader = (warp & 3) == 0;        // this warp issues the dQ reduce-adds
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t colS = w * 128, colDP = w * 128 + 64;
    const int kpos = k_tile * kTile + r;
    const bool k_valid = kpos < p.L;
    const int kb = k_valid ? kpos / p.M : -1;
    const float sl2 = p.scale_log2;
    uint8_t* xbase = smem + Lay::kX + w * Lay::kXBytes;
    float* stage = reinterpret_cast<float*>(smem + Lay::kStage + w * Lay::kStageBytes);
    const bool k_ragged = (k_tile + 1) * kTile > p.L;
    QWalk wk;
    wk.start(segs, n_segs);
    bool ok = true;
    int uses = 0;  // dQ staging uses of this stream
    for (int s = w; s < n_sub; s += 2, wk.next()) {
      const int k = s >> 1;
      const int qs = wk.stream;
      const int h = kvh * p.G + wk.g;
      const int q0 = wk.t * kTile + w * kSub;
      const int qst = s % kQStages;
      if (!mbar_wait_warp(&bars[C_S_FULL + w], k & 1, p.status, &abort_flag) ||
          !mbar_wait_warp(&bars[C_Q_FULL + qst], (s / kQStages) & 1, p.status, &abort_flag) ||
          (k > 0 && !mbar_wait_warp(&bars[C_X_FREE + w], (k - 1) & 1, p.status, &abort_flag))) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const float* lse = reinterpret_cast<const float*>(smem + Lay::kStat + qst * Lay::kStatBytes);
      const float* Dq = lse + kSub;
      const bool masked = (wk.flags & 1) || k_ragged || (q0 + kSub > p.L);
      // ---- P^T = exp(S^T scale - LSE), written back to TMEM as bf16 pairs
      float pr[kSub];
      tmem_ld32x2(tmem + lane_base + colS, tmem + lane_base + colS + 32, pr, pr + 32);
      if (masked) {
        // allowed query positions of this key row form one range [lo, hi)
        int lo, hi;
        allowed_query_range(qs, k_stream, kb, p.M, p.L, k_valid, lo, hi);
        lo -= q0;
        hi -= q0;
#pragma unroll
        for (int c = 0; c < kSub; ++c) {
          const float pv = ex2_approx(fmaf(pr[c], sl2, -lse[c] * kLog2e));
          pr[c] = (c >= lo && c < hi) ? pv : 0.f;
        }
      } else {
#pragma unroll
        for (int c = 0; c < kSub; ++c) pr[c] = ex2_approx(fmaf(pr[c], sl2, -lse[c] * kLog2e));
      }
      {
        float packed[32];
#pragma unroll
        for (int c = 0; c < 32; ++c) packed[c] = __uint_as_float(pack_bf16x2(pr[2 * c], pr[2 * c + 1]));
        tmem_st32(tmem + lane_base + colS, packed);
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_P_READY + w]);
      // ---- dS^T = P^T o (dP^T - D) into the shared tile
      if (!mbar_wait_warp(&bars[C_DP_FULL + w], k & 1, p.status, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      {
        float a[32], b[32];
        tmem_ld32x2(tmem + lane_base + colDP, tmem + lane_base + colDP + 32, a, b);
#pragma unroll
        for (int chunk = 0; chunk < kSub / 8; ++chunk) {
          const float* dp = (chunk < 4) ? a + chunk * 8 : b + (chunk - 4) * 8;
          const int c0 = chunk * 8;
          uint4 v;
          v.x = pack_bf16x2(pr[c0 + 0] * (dp[0] - Dq[c0 + 0]), pr[c0 + 1] * (dp[1] - Dq[c0 + 1]));
          v.y = pack_bf16x2(pr[c0 + 2] * (dp[2] - Dq[c0 + 2]), pr[c0 + 3] * (dp[3] - Dq[c0 + 3]));
          v.z = pack_bf16x2(pr[c0 + 4] * (dp[4] - Dq[c0 + 4]), pr[c0 + 5] * (dp[5] - Dq[c0 + 5]));
          v.w = pack_bf16x2(pr[c0 + 6] * (dp[6] - Dq[c0 + 6]), pr[c0 + 7] * (dp[7] - Dq[c0 + 7]));
          *reinterpret_cast<uint4*>(xbase + sw128_offset(r, chunk)) = v;
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_DS_READY + w]);
      // ---- dQ^T: thread r owns head-dim row r of the 64 query columns
      if (!mbar_wait_warp(&bars[C_DQ_FULL + w], k & 1, p.status, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      float dq[kSub];
      tmem_ld32x2(tmem + lane_base + colDP, tmem + lane_base + colDP + 32, dq, dq + 32);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_DQ_FREE + w]);
      // stage 32 query rows at a time ([row][d] fp32) and reduce-add them
#pragma unroll
      for (int half = 0; half < kSub / kStageRows; ++half, ++uses) {
        if (uses > 0 &&
            !mbar_wait_warp(&bars[C_STAGE_FREE + w], (uses - 1) & 1, p.status, &abort_flag)) {
          ok = false;
          break;
        }
        if (r < D) {
#pragma unroll
          for (int c = 0; c < kStageRows; ++c) stage[c * D + r] = dq[half * kStageRows + c];
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars[C_STAGE_FULL + w]);
        if (leader) {
          if (!mbar_wait_warp(&bars[C_STAGE_FULL + w], uses & 1, p.status, &abort_flag)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            tma_reduce_add_3d(&tm_dqacc, stage, h * D, q0 + half * kStageRows, qs * p.batch + bz);
            bulk_commit_group();
            bulk_wait_group_read<0>();
            mbar_arrive(&bars[C_STAGE_FREE + w]);
          }
          __syncwarp();
        }
      }
      if (!ok) break;
    }
    if (leader && lane == 0) bulk_wait_group<0>();  // reduce-adds complete before exit
    // ---- epilogue (stream 0): dV, dK rows of this key tile
    if (w == 0) {
      __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(k_stream ? p.dv[1] : p.dv[0]) +
                          ((static_cast<int64_t>(bz) * p.L + kpos) * p.Hkv + kvh) * D;
      __nv_bfloat16* dk = static_cast<__nv_bfloat16*>(k_stream ? p.dk[1] : p.dk[0]) +
                          ((static_cast<int64_t>(bz) * p.L + kpos) * p.Hkv + kvh) * D;
      if (n_sub == 0) {
        if (k_valid) {
          for (int c = 0; c < D; c += 8) {
            *reinterpret_cast<uint4*>(dv + c) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(dk + c) = make_uint4(0, 0, 0, 0);
          }
        }
      } else if (ok && mbar_wait_warp(&bars[C_ACC_DONE], 0, p.status, &abort_flag)) {
        tc_fence_after_sync();
#pragma unroll 1
        for (int half = 0; half < 2; ++half) {
          __nv_bfloat16* dstp = half ? dk : dv;
          const uint32_t col = half ? Lay::kColDK : Lay::kColDV;
          const float mul = half ? p.scale : 1.f;
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            float v[32];
            tmem_ld32(tmem + lane_base + col + ch * 32, v);
            if (k_valid) {
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
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(bwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kDynSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t grid = static_cast<int64_t>(n_tasks) * p.Hkv * p.batch;
  if (grid <= 0) return cudaSuccess;
  bwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, Lay::kDynSmem, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], maps[8], maps[9],
      maps[10], p);
  return cudaGetLastError();
}

// Rows of one TMA box for the query-side maps (Q, dO) and the LSE/D maps.
int bwd_query_box_rows() { return kSub; }
// Query rows of one dQ reduce-add box.
int bwd_dq_box_rows() { return kStageRows; }

// maps: q_clean, q_corr, k_clean, k_corr, v_clean, v_corr, do_clean, do_corr
//       (query-side maps with 64-row boxes), lse ({L, batch*2*Hq} fp32) and
//       dsum ({L, 2*batch*Hq} fp32) with 64-position boxes, dq_acc
//       ({Hq*d, L, 2*batch} fp32, box {d, 32, 1}, no swizzle)
cudaError_t launch_bwd(int d, const CUtensorMap* maps, const BwdParams& p, int n_tasks,
                       cudaStream_t stream) {
  if (d == 128) return launch_bwd_d<128>(maps, p, n_tasks, stream);
  return launch_bwd_d<64>(maps, p, n_tasks, stream);
}

}  // namespace csbp
