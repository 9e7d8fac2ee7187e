// Fused two-copy block-diffusion attention, forward, for sm_103a.
//
// Computes, per query row of either copy, softmax(scale * q K^T + mask) V over
// exactly the keys the block-diffusion mask allows ("CSBP 完全拆解" blog,
// section "CSBP：BP 管损坏块，CP 管干净上下文": O_b = Attn(Q_b, [K_b; K^clean_<b],
// [V_b; V^clean_<b]); clean queries block-causal over the clean copy), and the
// row's natural-log softmax denominator (LSE).  Partial mode writes one
// normalised fp32 partial per key part for the exact LSE merge of the
// section "在线 softmax 合并：为什么分两段算仍是同一个注意力".
//
// One CTA owns one 128-row query tile of one (batch, query head) and walks
// the key-tile segments of its work-list task.  Roles (256 threads):
//   warp 0 lane 0  TMA producer: Q once, then K_j / V_j into 2-stage rings
//   warp 1 lane 0  MMA issuer:   S_j = Q K_j^T into TMEM (double buffered),
//                                O += P_{j-1} V_{j-1} into TMEM
//   warps 4..7     softmax: thread t owns query row t (TMEM lane t); reads
//                  S_j with tcgen05.ld, masks partial tiles, keeps a running
//                  reference max, writes P_j (bf16) to shared memory in the
//                  128B-swizzled K-major layout the PV MMA reads, and
//                  rescales the TMEM accumulator only when the row max grows
//                  by more than 2^8 (exact: O and l share the reference).
// TMEM columns: S buffers at 0 and 128, O at 256 (512 allocated).
#include <cuda.h>
#include <cuda_runtime.h>

#include "csbp_internal.h"
#include "ptx_sm100.cuh"

namespace csbp {

namespace {

constexpr int kThreads = 256;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;     // Q/K/V tile (bf16)
  static constexpr int kBoxBytes = kTile * 64 * 2;     // one 64-column TMA box
  static constexpr int kPBytes = kTile * kTile * 2;    // P tile (bf16)
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;           // 2 stages
  static constexpr int kV = kK + 2 * kTileBytes;       // 2 stages
  static constexpr int kP = kV + 2 * kTileBytes;       // 2 buffers
  static constexpr int kBytes = kP + 2 * kPBytes;
  static constexpr int kDynSmem = kBytes + 1024;       // + alignment slack
};

enum FwdBar {
  B_Q_FULL = 0,
  B_K_FULL,            // [2]
  B_V_FULL = B_K_FULL + 2,
  B_K_EMPTY = B_V_FULL + 2,
  B_V_EMPTY = B_K_EMPTY + 2,
  B_S_FULL = B_V_EMPTY + 2,
  B_S_FREE = B_S_FULL + 2,
  B_P_FULL = B_S_FREE + 2,
  B_P_EMPTY = B_P_FULL + 2,
  B_DRAIN = B_P_EMPTY + 2,
  B_COUNT
};

// Sequential walk over the key tiles of a task's segments.
struct TileWalk {
  const int32_t* seg;
  int remaining_segs;
  int stream, t, end, flags;
  __device__ void start(const int32_t* s, int n) {
    seg = s;
    remaining_segs = n;
    end = 0;
    t = 0;
    advance_segment();
  }
  __device__ void advance_segment() {
    if (remaining_segs <= 0) return;
    stream = seg[0];
    t = seg[1];
    end = seg[2];
    flags = seg[3];
    seg += kSegWords;
    --remaining_segs;
  }
  __device__ void next() {
    ++t;
    if (t >= end) advance_segment();
  }
};

// Key positions [lo, hi) of copy k_stream that a query of block qb of copy
// q_stream may read: clean queries read clean keys of blocks <= qb;
// corrupted queries read clean keys of blocks < qb and the corrupted keys of
// their own block.
__device__ __forceinline__ void allowed_key_range(int q_stream, int k_stream, int qb, int M, int L,
                                                  bool row_valid, int& lo, int& hi) {
  lo = 0;
  if (!row_valid || (q_stream == 0 && k_stream == 1)) {
    hi = 0;
    return;
  }
  if (q_stream == 0) {
    hi = (qb + 1) * M;
  } else if (k_stream == 0) {
    hi = qb * M;
  } else {
    lo = qb * M;
    hi = (qb + 1) * M;
  }
  hi = min(hi, L);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    fwd_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
               const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_k1,
               const __grid_constant__ CUtensorMap tm_v0, const __grid_constant__ CUtensorMap tm_v1,
               const FwdParams p) {
  using Lay = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  __shared__ uint64_t bars[B_COUNT];
  __shared__ uint32_t tmem_base_sh;
  __shared__ int abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- decode the unit: (task, batch, query head)
  const int hb = p.Hq * p.batch;
  const int task = blockIdx.x / hb;
  const int rem = blockIdx.x - task * hb;
  const int bz = rem / p.Hq;
  const int h = rem - bz * p.Hq;
  const int kvh = h / p.G;
  const int32_t* tw = p.tasks + static_cast<int64_t>(task) * kTaskWords;
  const int q_stream = tw[0];
  const int q_tile = tw[1];
  const int part = tw[2];
  const int32_t* segs = p.segs + static_cast<int64_t>(tw[3]) * kSegWords;
  const int n_segs = tw[4];
  const int n_tiles = tw[5];

  if (threadIdx.x == 0) {
    for (int i = 0; i < B_COUNT; ++i) {
      const bool per_warp = (i >= B_S_FREE && i < B_S_FREE + 2) || (i >= B_P_FULL && i < B_P_FULL + 2);
      mbar_init(&bars[i], per_warp ? 4 : 1);  // softmax warps arrive once each
    }
    abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(&tmem_base_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = tmem_base_sh;

  const uint32_t sQ = smem_u32(smem + Lay::kQ);
  const uint32_t sK = smem_u32(smem + Lay::kK);
  const uint32_t sV = smem_u32(smem + Lay::kV);
  const uint32_t sP = smem_u32(smem + Lay::kP);

  if (warp == 0 && lane == 0) {
    // ===================== TMA producer
    const void* tq = q_stream ? static_cast<const void*>(&tm_q1) : static_cast<const void*>(&tm_q0);
    prefetch_tmap(tq);
    prefetch_tmap(&tm_k0);
    prefetch_tmap(&tm_k1);
    prefetch_tmap(&tm_v0);
    prefetch_tmap(&tm_v1);
    mbar_arrive_expect_tx(&bars[B_Q_FULL], Lay::kTileBytes);
#pragma unroll
    for (int c = 0; c < D / 64; ++c)
      tma_load_3d(smem + Lay::kQ + c * Lay::kBoxBytes, tq, &bars[B_Q_FULL], h * D + c * 64,
                  q_tile * kTile, bz);
    TileWalk w;
    w.start(segs, n_segs);
    int nk = 0, nv = 0;  // K / V tiles whose loads were issued
    bool ok = true;
    for (int j = 0; j < n_tiles && ok; ++j, w.next()) {
      const int b = j & 1;
      const void* tk = w.stream ? static_cast<const void*>(&tm_k1) : static_cast<const void*>(&tm_k0);
      const void* tv = w.stream ? static_cast<const void*>(&tm_v1) : static_cast<const void*>(&tm_v0);
      if (j >= 2) ok = mbar_wait(&bars[B_K_EMPTY + b], ((j - 2) >> 1) & 1, p.status, &abort_flag);
      if (!ok) break;
      mbar_arrive_expect_tx(&bars[B_K_FULL + b], Lay::kTileBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + Lay::kK + b * Lay::kTileBytes + c * Lay::kBoxBytes, tk,
                    &bars[B_K_FULL + b], kvh * D + c * 64, w.t * kTile, bz);
      nk = j + 1;
      if (j >= 2) ok = mbar_wait(&bars[B_V_EMPTY + b], ((j - 2) >> 1) & 1, p.status, &abort_flag);
      if (!ok) break;
      mbar_arrive_expect_tx(&bars[B_V_FULL + b], Lay::kTileBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + Lay::kV + b * Lay::kTileBytes + c * Lay::kBoxBytes, tv,
                    &bars[B_V_FULL + b], kvh * D + c * 64, w.t * kTile, bz);
      nv = j + 1;
    }
    if (!ok) {
      // drain: wait (ignoring the abort flag) for the loads already issued
      // (at most the last two tiles of each ring can still be in flight)
      mbar_wait(&bars[B_Q_FULL], 0, nullptr, nullptr, 200000000ull);
      for (int j = (nk > 2 ? nk - 2 : 0); j < nk; ++j)
        mbar_wait(&bars[B_K_FULL + (j & 1)], (j >> 1) & 1, nullptr, nullptr, 200000000ull);
      for (int j = (nv > 2 ? nv - 2 : 0); j < nv; ++j)
        mbar_wait(&bars[B_V_FULL + (j & 1)], (j >> 1) & 1, nullptr, nullptr, 200000000ull);
    }
  } else if (warp == 1 && lane == 0) {
    // ===================== MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, false, true);
    bool ok = mbar_wait(&bars[B_Q_FULL], 0, p.status, &abort_flag);
    const uint64_t q_desc = sdesc_sw128(sQ, 16, 1024);  // Q as K-major A
    auto issue_pv = [&](int i) -> bool {
      const int c = i & 1;
      if (!mbar_wait(&bars[B_P_FULL + c], (i >> 1) & 1, p.status, &abort_flag)) return false;
      if (!mbar_wait(&bars[B_V_FULL + c], (i >> 1) & 1, p.status, &abort_flag)) return false;
      tc_fence_after_sync();
      const uint64_t pa = sdesc_sw128(sP + c * Lay::kPBytes, 16, 1024);               // P, K-major A
      const uint64_t vb = sdesc_sw128(sV + c * Lay::kTileBytes, Lay::kBoxBytes, 1024);  // V, MN-major B
      const uint32_t acc0 = i > 0 ? 1u : 0u;
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k)
        umma_bf16_ss(tmem + 256, sdesc_step(pa, (k >> 2) * Lay::kBoxBytes + (k & 3) * 32),
                     sdesc_step(vb, k * 2048), idesc_pv, k > 0 ? 1u : acc0);
      umma_commit(&bars[B_P_EMPTY + c]);
      umma_commit(&bars[B_V_EMPTY + c]);
      return true;
    };
    for (int j = 0; j < n_tiles && ok; ++j) {
      const int b = j & 1;
      ok = mbar_wait(&bars[B_K_FULL + b], (j >> 1) & 1, p.status, &abort_flag);
      if (ok && j >= 2) ok = mbar_wait(&bars[B_S_FREE + b], ((j - 2) >> 1) & 1, p.status, &abort_flag);
      if (!ok) break;
      tc_fence_after_sync();
      const uint64_t k_desc = sdesc_sw128(sK + b * Lay::kTileBytes, 16, 1024);  // K, K-major B
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * Lay::kBoxBytes + (k & 3) * 32;
        umma_bf16_ss(tmem + b * 128, sdesc_step(q_desc, off), sdesc_step(k_desc, off), idesc_s,
                     k > 0 ? 1u : 0u);
      }
      umma_commit(&bars[B_S_FULL + b]);
      umma_commit(&bars[B_K_EMPTY + b]);
      if (j >= 1) ok = issue_pv(j - 1);
    }
    if (ok) issue_pv(n_tiles - 1);
    // drain every MMA this thread issued before the CTA may free TMEM
    umma_commit(&bars[B_DRAIN]);
    mbar_wait(&bars[B_DRAIN], 0, nullptr, nullptr, 500000000ull);
  } else if (warp >= 4) {
    // ===================== softmax warpgroup
    const int row = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const int64_t qpos = static_cast<int64_t>(q_tile) * kTile + row;
    const bool row_valid = qpos < p.L;
    const int qb = row_valid ? static_cast<int>(qpos) / p.M : -1;
    const float sl2 = p.scale_log2;
    float m_ref = -INFINITY;
    float l = 0.f;
    TileWalk w;
    w.start(segs, n_segs);
    bool ok = true;
    uint8_t* sPbase = smem + Lay::kP;
    for (int j = 0; j < n_tiles; ++j, w.next()) {
      const int b = j & 1;
      if (!mbar_wait_warp(&bars[B_S_FULL + b], (j >> 1) & 1, p.status, &abort_flag)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      float s[kTile];
#pragma unroll
      for (int c = 0; c < kTile / 32; ++c) tmem_ld32(tmem + lane_base + b * 128 + c * 32, s + c * 32);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_S_FREE + b]);

      const bool ragged = (static_cast<int64_t>(w.t) + 1) * kTile > p.L;
      float mx = -INFINITY;
      if ((w.flags & 1) || ragged || !row_valid) {
        // the allowed keys of this query row form one range [lo, hi)
        int lo, hi;
        allowed_key_range(q_stream, w.stream, qb, p.M, p.L, row_valid, lo, hi);
        lo -= w.t * kTile;
        hi -= w.t * kTile;
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          s[c] = (c >= lo && c < hi) ? s[c] * sl2 : -INFINITY;
          mx = fmaxf(mx, s[c]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < kTile; ++c) {
          s[c] *= sl2;
          mx = fmaxf(mx, s[c]);
        }
      }
      const float m_new = fmaxf(m_ref, mx);
      const bool need = m_new > m_ref + kRescaleThreshold;  // false while both are -inf
      if (j > 0 && __any_sync(0xffffffffu, need)) {
        // O holds PV_0..PV_{j-1} scaled by the old reference: wait for PV_{j-1}
        if (!mbar_wait_warp(&bars[B_P_EMPTY + ((j - 1) & 1)], ((j - 1) >> 1) & 1, p.status, &abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const float alpha = need ? exp2f(m_ref - m_new) : 1.f;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_base + 256 + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tmem + lane_base + 256 + c * 32, o);
        }
      }
      if (need) {
        l *= exp2f(m_ref - m_new);  // 0 when m_ref was -inf
        m_ref = m_new;
      }
      const float mref_safe = (m_ref == -INFINITY) ? 0.f : m_ref;
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kTile; ++c) {
        s[c] = ex2_approx(s[c] - mref_safe);
        rs += s[c];
      }
      l += rs;
      if (j >= 2 && !mbar_wait_warp(&bars[B_P_EMPTY + b], ((j - 2) >> 1) & 1, p.status, &abort_flag)) {
        ok = false;
        break;
      }
      uint8_t* pb = sPbase + b * Lay::kPBytes;
#pragma unroll
      for (int ch = 0; ch < kTile / 8; ++ch) {
        uint4 v;
        v.x = pack_bf16x2(s[ch * 8 + 0], s[ch * 8 + 1]);
        v.y = pack_bf16x2(s[ch * 8 + 2], s[ch * 8 + 3]);
        v.z = pack_bf16x2(s[ch * 8 + 4], s[ch * 8 + 5]);
        v.w = pack_bf16x2(s[ch * 8 + 6], s[ch * 8 + 7]);
        *reinterpret_cast<uint4*>(pb + (ch >> 3) * Lay::kBoxBytes + sw128_offset(row, ch & 7)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[B_P_FULL + b]);
    }
    // ---- epilogue: wait for the last PV, normalise, store
    if (ok && mbar_wait_warp(&bars[B_P_EMPTY + ((n_tiles - 1) & 1)], ((n_tiles - 1) >> 1) & 1, p.status,
                        &abort_flag)) {
      tc_fence_after_sync();
      const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
      const float lse = (l > 0.f) ? (m_ref + log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (p.partial_mode) {
        const int64_t prow = ((static_cast<int64_t>(part) * 2 + q_stream) * p.batch + bz);
        float* dst = p.part_o + (prow * p.L + qpos) * p.Hq * D + static_cast<int64_t>(h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_base + 256 + c * 32, o);
          if (row_valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
              *reinterpret_cast<float4*>(dst + c * 32 + i) =
                  make_float4(o[i] * inv_l, o[i + 1] * inv_l, o[i + 2] * inv_l, o[i + 3] * inv_l);
          }
        }
        if (row_valid) p.part_lse[(prow * p.Hq + h) * p.L + qpos] = lse;
      } else {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(q_stream ? p.o[1] : p.o[0]) +
                             ((static_cast<int64_t>(bz) * p.L + qpos) * p.Hq + h) * D;
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tmem + lane_base + 256 + c * 32, o);
          if (row_valid) {
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              v.x = pack_bf16x2(o[i] * inv_l, o[i + 1] * inv_l);
              v.y = pack_bf16x2(o[i + 2] * inv_l, o[i + 3] * inv_l);
              v.z = pack_bf16x2(o[i + 4] * inv_l, o[i + 5] * inv_l);
              v.w = pack_bf16x2(o[i + 6] * inv_l, o[i + 7] * inv_l);
              *reinterpret_cast<uint4*>(dst + c * 32 + i) = v;
            }
          }
        }
        if (row_valid)
          p.lse[((static_cast<int64_t>(bz) * 2 + q_stream) * p.Hq + h) * p.L + qpos] = lse;
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
static cudaError_t launch_fwd_d(const CUtensorMap* maps, const FwdParams& p, int n_tasks,
                                cudaStream_t stream) {
  using Lay = FwdLayout<D>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Lay::kDynSmem);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  const int64_t grid = static_cast<int64_t>(n_tasks) * p.Hq * p.batch;
  if (grid <= 0) return cudaSuccess;
  fwd_kernel<D><<<static_cast<unsigned>(grid), kThreads, Lay::kDynSmem, stream>>>(
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], p);
  return cudaGetLastError();
}

// maps: q_clean, q_corr, k_clean, k_corr, v_clean, v_corr
cudaError_t launch_fwd(int d, const CUtensorMap* maps, const FwdParams& p, int n_tasks,
                       cudaStream_t stream) {
  if (d == 128) return launch_fwd_d<128>(maps, p, n_tasks, stream);
  return launch_fwd_d<64>(maps, p, n_tasks, stream);
}

}  // namespace csbp
