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
// (query head of the GQA group, query tile) its work-list task lists, so dK/dV
// accumulate in TMEM for the whole group and are written once.  Roles:
//   warp 0 lane 0  TMA producer: K, V once; Q (2 stages) and dO per step
//   warp 1 lane 0  MMA issuer:   S^T = K Q^T, dP^T = V dO^T; dV += P^T dO;
//                                dK += dS^T Q; dQ_tile = dS K
//   warps 4..7     thread t owns key row t for S^T/dP^T/dV/dK and query row
//                  t for the dQ tile; P^T and then dS^T go through one
//                  128B-swizzled shared tile that serves as K-major A operand
//                  (dV, dK) and, read transposed, as MN-major A operand (dQ).
//                  dQ tiles are added into an fp32 accumulator with vector
//                  atomics.
// TMEM columns: S^T (later the dQ tile) at 0, dP^T at 128, dV at 256, dK at 384.
#include <cuda.h>
#include <cuda_runtime.h>

#include "csbp_internal.h"
#include "ptx_sm100.cuh"

namespace csbp {

namespace {

constexpr int kThreads = 256;

template <int D>
struct BwdLayout {
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kBoxBytes = kTile * 64 * 2;
  static constexpr int kXBytes = kTile * kTile * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;        // 2 stages
  static constexpr int kDO = kQ + 2 * kTileBytes;   // 1 stage
  static constexpr int kX = kDO + kTileBytes;       // P^T, then dS^T
  static constexpr int kStat = kX + kXBytes;        // [4 warps][lse2 | D][128] fp32
  static constexpr int kBytes = kStat + 4 * 2 * kTile * 4;
  static constexpr int kDynSmem = kBytes + 1024;
  static constexpr uint32_t kColDV = 256;
  static constexpr uint32_t kColDK = 256 + (D > 64 ? 128 : 64);
};

enum BwdBar {
  C_KV_FULL = 0,
  C_Q_FULL,  // [2]
  C_Q_EMPTY = C_Q_FULL + 2,
  C_DO_FULL = C_Q_EMPTY + 2,
  C_DO_EMPTY,
  C_S_FULL,
  C_P_READY,
  C_X_FREE,
  C_DS_READY,
  C_X_FREE2,
  C_DQ_FULL,
  C_DQ_FREE,
  C_ACC_DONE,
  C_DRAIN,
  C_COUNT
};

// Walk over (query head in group, segment, query tile) of a backward task.
struct QWalk {
  const int32_t* seg0;
  int n_segs, g, G, si, t, end, stream, flags;
  __device__ void load_seg() {
    const int32_t* s = seg0 + si * kSegWords;
    stream = s[0];
    t = s[1];
    end = s[2];
    flags = s[3];
  }
  __device__ void start(const int32_t* s, int n, int groups) {
    seg0 = s;
    n_segs = n;
    G = groups;
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

__device__ __forceinline__ bool mask_allows(int q_stream, int k_stream, int qb, int kb) {
  if (q_stream == 0) return k_stream == 0 && kb <= qb;
  return k_stream == 0 ? (kb < qb) : (kb == qb);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_kernel(const __grid_constant__ CUtensorMap tm_q0, const __grid_constant__ CUtensorMap tm_q1,
               const __grid_constant__ CUtensorMap tm_k0, const __grid_constant__ CUtensorMap tm_k1,
               const __grid_constant__ CUtensorMap tm_v0, const __grid_constant__ CUtensorMap tm_v1,
               const __grid_constant__ CUtensorMap tm_do0,
               const __grid_constant__ CUtensorMap tm_do1, const BwdParams p) {
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
  const int n_iters = tw[5] * p.G;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C_COUNT; ++i) {
      const bool per_warp = (i == C_P_READY || i == C_DS_READY || i == C_DQ_FREE);
      mbar_init(&bars[i], per_warp ? 4 : 1);
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

  const uint32_t sK = smem_u32(smem + Lay::kK);
  const uint32_t sV = smem_u32(smem + Lay::kV);
  const uint32_t sQ = smem_u32(smem + Lay::kQ);
  const uint32_t sDO = smem_u32(smem + Lay::kDO);
  const uint32_t sX = smem_u32(smem + Lay::kX);

  if (n_iters > 0 && warp == 0 && lane == 0) {
    // ===================== TMA producer
    const void* tk = k_stream ? static_cast<const void*>(&tm_k1) : static_cast<const void*>(&tm_k0);
    const void* tv = k_stream ? static_cast<const void*>(&tm_v1) : static_cast<const void*>(&tm_v0);
    mbar_arrive_expect_tx(&bars[C_KV_FULL], 2 * Lay::kTileBytes);
#pragma unroll
    for (int c = 0; c < D / 64; ++c) {
      tma_load_3d(smem + Lay::kK + c * Lay::kBoxBytes, tk, &bars[C_KV_FULL], kvh * D + c * 64,
                  k_tile * kTile, bz);
      tma_load_3d(smem + Lay::kV + c * Lay::kBoxBytes, tv, &bars[C_KV_FULL], kvh * D + c * 64,
                  k_tile * kTile, bz);
    }
    QWalk w;
    w.start(segs, n_segs, p.G);
    int nq = 0, ndo = 0;
    bool ok = true;
    for (int i = 0; i < n_iters; ++i, w.next()) {
      const int st = i & 1;
      const int h = kvh * p.G + w.g;
      const void* tq = w.stream ? static_cast<const void*>(&tm_q1) : static_cast<const void*>(&tm_q0);
      const void* td = w.stream ? static_cast<const void*>(&tm_do1) : static_cast<const void*>(&tm_do0);
      if (i >= 2) ok = mbar_wait(&bars[C_Q_EMPTY + st], ((i - 2) >> 1) & 1, p.status, &abort_flag);
      if (!ok) break;
      mbar_arrive_expect_tx(&bars[C_Q_FULL + st], Lay::kTileBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + Lay::kQ + st * Lay::kTileBytes + c * Lay::kBoxBytes, tq,
                    &bars[C_Q_FULL + st], h * D + c * 64, w.t * kTile, bz);
      nq = i + 1;
      if (i >= 1) ok = mbar_wait(&bars[C_DO_EMPTY], (i - 1) & 1, p.status, &abort_flag);
      if (!ok) break;
      mbar_arrive_expect_tx(&bars[C_DO_FULL], Lay::kTileBytes);
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tma_load_3d(smem + Lay::kDO + c * Lay::kBoxBytes, td, &bars[C_DO_FULL], h * D + c * 64,
                    w.t * kTile, bz);
      ndo = i + 1;
    }
    if (!ok) {
      mbar_wait(&bars[C_KV_FULL], 0, nullptr, nullptr, 200000000ull);
      for (int i = (nq > 2 ? nq - 2 : 0); i < nq; ++i)
        mbar_wait(&bars[C_Q_FULL + (i & 1)], (i >> 1) & 1, nullptr, nullptr, 200000000ull);
      if (ndo > 0) mbar_wait(&bars[C_DO_FULL], (ndo - 1) & 1, nullptr, nullptr, 200000000ull);
    }
  } else if (n_iters > 0 && warp == 1 && lane == 0) {
    // ===================== MMA issuer
    constexpr uint32_t idesc_sq = idesc_bf16_f32(128, 128, false, false);  // S^T, dP^T
    constexpr uint32_t idesc_kd = idesc_bf16_f32(128, D, false, true);     // dV, dK
    constexpr uint32_t idesc_q = idesc_bf16_f32(128, D, true, true);       // dQ
    bool ok = mbar_wait(&bars[C_KV_FULL], 0, p.status, &abort_flag);
    for (int i = 0; i < n_iters && ok; ++i) {
      const int st = i & 1;
      const uint32_t q_s = sQ + st * Lay::kTileBytes;
      ok = mbar_wait(&bars[C_Q_FULL + st], (i >> 1) & 1, p.status, &abort_flag) &&
           mbar_wait(&bars[C_DO_FULL], i & 1, p.status, &abort_flag) &&
           (i == 0 || mbar_wait(&bars[C_DQ_FREE], (i - 1) & 1, p.status, &abort_flag));
      if (!ok) break;
      tc_fence_after_sync();
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * Lay::kBoxBytes + (k & 3) * 32;
        umma_bf16_ss(tmem + 0, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(q_s + off, 16, 1024),
                     idesc_sq, k > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * Lay::kBoxBytes + (k & 3) * 32;
        umma_bf16_ss(tmem + 128, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024),
                     idesc_sq, k > 0 ? 1u : 0u);
      }
      umma_commit(&bars[C_S_FULL]);
      if (!mbar_wait(&bars[C_P_READY], i & 1, p.status, &abort_flag)) break;
      tc_fence_after_sync();
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k) {
        const uint64_t ad = sdesc_sw128(sX + (k >> 2) * Lay::kBoxBytes + (k & 3) * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(sDO + k * 2048, Lay::kBoxBytes, 1024);
        umma_bf16_ss(tmem + Lay::kColDV, ad, bd, idesc_kd, (i > 0 || k > 0) ? 1u : 0u);
      }
      umma_commit(&bars[C_X_FREE]);
      umma_commit(&bars[C_DO_EMPTY]);
      if (!mbar_wait(&bars[C_DS_READY], i & 1, p.status, &abort_flag)) break;
      tc_fence_after_sync();
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k) {
        const uint64_t ad = sdesc_sw128(sX + (k >> 2) * Lay::kBoxBytes + (k & 3) * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(q_s + k * 2048, Lay::kBoxBytes, 1024);
        umma_bf16_ss(tmem + Lay::kColDK, ad, bd, idesc_kd, (i > 0 || k > 0) ? 1u : 0u);
      }
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k) {
        const uint64_t ad = sdesc_sw128(sX + k * 2048, Lay::kBoxBytes, 1024);
        const uint64_t bd = sdesc_sw128(sK + k * 2048, Lay::kBoxBytes, 1024);
        umma_bf16_ss(tmem + 0, ad, bd, idesc_q, k > 0 ? 1u : 0u);
      }
      umma_commit(&bars[C_DQ_FULL]);
      umma_commit(&bars[C_Q_EMPTY + st]);
      umma_commit(&bars[C_X_FREE2]);
    }
    umma_commit(&bars[C_ACC_DONE]);
    umma_commit(&bars[C_DRAIN]);
    mbar_wait(&bars[C_DRAIN], 0, nullptr, nullptr, 500000000ull);
  } else if (warp >= 4) {
    // ===================== compute warpgroup
    const int r = threadIdx.x - 128;
    const uint32_t lane_base = static_cast<uint32_t>((warp - 4) * 32) << 16;
    const int kpos = k_tile * kTile + r;
    const bool k_valid = kpos < p.L;
    const int kb = k_valid ? kpos / p.M : -1;
    const float sl2 = p.scale_log2;
    float* stat = reinterpret_cast<float*>(smem + Lay::kStat);
    uint8_t* xbase = smem + Lay::kX;
    const bool k_ragged = (k_tile + 1) * kTile > p.L;
    QWalk w;
    w.start(segs, n_segs, p.G);
    bool ok = true;
    for (int i = 0; i < n_iters; ++i, w.next()) {
      const int h = kvh * p.G + w.g;
      const int qs = w.stream;
      const int q0 = w.t * kTile;
      // stage LSE (log2 units) and D of the 128 query columns in this warp's
      // own slice (warp-local sync only)
      float* lse2 = stat + (warp - 4) * 2 * kTile;
      float* Dq = lse2 + kTile;
      {
        const int64_t rbase = ((static_cast<int64_t>(bz) * 2 + qs) * p.Hq + h) * p.L;
        const int64_t dbase = ((static_cast<int64_t>(qs) * p.batch + bz) * p.Hq + h) * p.L;
        __syncwarp();
#pragma unroll
        for (int e = 0; e < kTile / 32; ++e) {
          const int c = e * 32 + lane;
          const int qpos = q0 + c;
          lse2[c] = (qpos < p.L) ? p.lse[rbase + qpos] * 1.4426950408889634f : INFINITY;
          Dq[c] = (qpos < p.L) ? p.Dsum[dbase + qpos] : 0.f;
        }
        __syncwarp();
      }
      if (!mbar_wait_warp(&bars[C_S_FULL], i & 1, p.status, &abort_flag)) { ok = false; break; }
      if (i > 0 && !mbar_wait_warp(&bars[C_X_FREE2], (i - 1) & 1, p.status, &abort_flag)) { ok = false; break; }
      tc_fence_after_sync();
      const bool masked = (w.flags & 1) || k_ragged || (q0 + kTile > p.L);
      uint32_t ds_pack[kTile / 2];
      int qb = q0 / p.M;
      int qr = q0 - qb * p.M;
#pragma unroll
      for (int ch = 0; ch < kTile / 32; ++ch) {
        float sv[32], dp[32];
        tmem_ld32(tmem + lane_base + 0 + ch * 32, sv);
        tmem_ld32(tmem + lane_base + 128 + ch * 32, dp);
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int c = ch * 32 + e;
          float pv = ex2_approx(sv[e] * sl2 - lse2[c]);
          if (masked) {
            const bool allow = k_valid && (q0 + c < p.L) && mask_allows(qs, k_stream, qb, kb);
            pv = allow ? pv : 0.f;
            if (++qr == p.M) {
              qr = 0;
              ++qb;
            }
          }
          sv[e] = pv;
          dp[e] = pv * (dp[e] - Dq[c]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int chunk = ch * 4 + k;  // 16-byte chunk of the 256-byte row
          uint4 v;
          v.x = pack_bf16x2(sv[k * 8 + 0], sv[k * 8 + 1]);
          v.y = pack_bf16x2(sv[k * 8 + 2], sv[k * 8 + 3]);
          v.z = pack_bf16x2(sv[k * 8 + 4], sv[k * 8 + 5]);
          v.w = pack_bf16x2(sv[k * 8 + 6], sv[k * 8 + 7]);
          *reinterpret_cast<uint4*>(xbase + (chunk >> 3) * Lay::kBoxBytes + sw128_offset(r, chunk & 7)) = v;
          ds_pack[chunk * 4 + 0] = pack_bf16x2(dp[k * 8 + 0], dp[k * 8 + 1]);
          ds_pack[chunk * 4 + 1] = pack_bf16x2(dp[k * 8 + 2], dp[k * 8 + 3]);
          ds_pack[chunk * 4 + 2] = pack_bf16x2(dp[k * 8 + 4], dp[k * 8 + 5]);
          ds_pack[chunk * 4 + 3] = pack_bf16x2(dp[k * 8 + 6], dp[k * 8 + 7]);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_P_READY]);
      if (!mbar_wait_warp(&bars[C_X_FREE], i & 1, p.status, &abort_flag)) { ok = false; break; }
#pragma unroll
      for (int chunk = 0; chunk < kTile / 8; ++chunk) {
        uint4 v = make_uint4(ds_pack[chunk * 4 + 0], ds_pack[chunk * 4 + 1], ds_pack[chunk * 4 + 2],
                             ds_pack[chunk * 4 + 3]);
        *reinterpret_cast<uint4*>(xbase + (chunk >> 3) * Lay::kBoxBytes + sw128_offset(r, chunk & 7)) = v;
      }
      fence_proxy_async_smem();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_DS_READY]);
      // ---- drain the dQ tile: this thread owns query row q0 + r
      if (!mbar_wait_warp(&bars[C_DQ_FULL], i & 1, p.status, &abort_flag)) { ok = false; break; }
      tc_fence_after_sync();
      {
        const int qpos = q0 + r;
        float* dst = p.dq_acc +
                     (((static_cast<int64_t>(qs) * p.batch + bz) * p.L + qpos) * p.Hq + h) * D;
#pragma unroll 1
        for (int ch = 0; ch < D / 32; ++ch) {
          float v[32];
          tmem_ld32(tmem + lane_base + 0 + ch * 32, v);
          if (qpos < p.L) {
#pragma unroll
            for (int e = 0; e < 32; e += 4)
              atomicAdd(reinterpret_cast<float4*>(dst + ch * 32 + e),
                        make_float4(v[e], v[e + 1], v[e + 2], v[e + 3]));
          }
        }
      }
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[C_DQ_FREE]);
    }
    // ---- epilogue: dV, dK rows of this key tile
    __nv_bfloat16* dv = static_cast<__nv_bfloat16*>(k_stream ? p.dv[1] : p.dv[0]) +
                        ((static_cast<int64_t>(bz) * p.L + kpos) * p.Hkv + kvh) * D;
    __nv_bfloat16* dk = static_cast<__nv_bfloat16*>(k_stream ? p.dk[1] : p.dk[0]) +
                        ((static_cast<int64_t>(bz) * p.L + kpos) * p.Hkv + kvh) * D;
    if (n_iters == 0) {
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
        __nv_bfloat16* dst = half ? dk : dv;
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
              *reinterpret_cast<uint4*>(dst + ch * 32 + e) = u;
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
      maps[0], maps[1], maps[2], maps[3], maps[4], maps[5], maps[6], maps[7], p);
  return cudaGetLastError();
}

// maps: q_clean, q_corr, k_clean, k_corr, v_clean, v_corr, do_clean, do_corr
cudaError_t launch_bwd(int d, const CUtensorMap* maps, const BwdParams& p, int n_tasks,
                       cudaStream_t stream) {
  if (d == 128) return launch_bwd_d<128>(maps, p, n_tasks, stream);
  return launch_bwd_d<64>(maps, p, n_tasks, stream);
}

}  // namespace csbp
