// Streamed LM-head cross-entropy (csbp_vocab_ce.h): a persistent tcgen05
// GEMM with three epilogues, and a row kernel, run chunk by chunk.
//
// Per chunk of C rows:
//   1. logits GEMM   Z = H_c W^T (M = C, N = V, K = Dm); the epilogue writes
//      fp32 Z and, per row and 256-column vocabulary tile, the running max and
//      sum of exp, and the target's logit when it falls in the tile;
//   2. row kernel    merges the partials into LSE and the loss, and writes
//      g = s (softmax - onehot) as bf16;
//   3. dH GEMM       dH_c = g W (M = C, N = Dm, K = V), bf16 out;
//   4. dW GEMM       dW (+)= g^T H_c (M = V, N = Dm, K = C), fp32 out
//      (trained head only; the first chunk stores, later chunks add).
//
// GEMM tile 128 x 256 with K steps of 64 (one 128-byte swizzle atom), 4
// stages of TMA-loaded operands, fp32 accumulators in TMEM double-buffered
// (2 x 256 columns) so a tile's epilogue overlaps the next tile's MMAs.
// Roles (256 threads): warp 0 lane 0 TMA producer, warp 1 lane 0 MMA issuer,
// warps 4-7 epilogue (one accumulator row = TMEM lane per thread).  One CTA
// per SM, persistent over tiles.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "csbp.h"
#include "csbp_internal.h"
#include "csbp_vocab_ce.h"
#include "ptx_sm100.cuh"

namespace csbp {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, kStages = 4;
constexpr int kGemmThreads = 256;
constexpr uint32_t kABytes = BM * BK * 2;        // 16 KB
constexpr uint32_t kBBytes = BN * BK * 2;        // 32 KB
constexpr uint32_t kChunkBytes = 64 * BK * 2;    // one 64 x 64 MN-major box (8 KB)
constexpr uint32_t kSmemA = 0;
constexpr uint32_t kSmemB = kStages * kABytes;
constexpr uint32_t kSmemBar = kSmemB + kStages * kBBytes;
enum {
  G_FULL = 0,
  G_EMPTY = G_FULL + kStages,
  G_ACC_FULL = G_EMPTY + kStages,
  G_ACC_EMPTY = G_ACC_FULL + 2,
  G_DRAIN = G_ACC_EMPTY + 2,
  G_COUNT
};
constexpr uint32_t kSmemMisc = kSmemBar + G_COUNT * 8;
constexpr uint32_t kSmemTotal = kSmemMisc + 16;
constexpr int kDefaultChunk = 8192;
constexpr int kRowThreads = 256;
constexpr uint64_t kDrainNs = 200000000ull;
constexpr float kLog2e = 1.4426950408889634f;

enum Epi { EPI_LOGITS = 0, EPI_BF16 = 1, EPI_F32 = 2 };

struct GemmParams {
  int32_t M, N, K;           // output rows, output columns, reduction length
  int32_t n_mt, n_nt, n_tiles, group_m;
  int* status;
  // EPI_LOGITS
  float* z;                  // fp32 [M][ldz]
  int64_t ldz;
  float2* part;              // [M][n_nt]: (max, sum of exp) of each column tile
  float* zt;                 // [M]: the target's logit
  const int32_t* target;     // [M]
  // EPI_BF16 / EPI_F32
  void* out;                 // bf16 or fp32 [M][ld_out]
  int64_t ld_out;
  int32_t accumulate;        // EPI_F32: add to the existing values
};

// Tiles are taken in groups of group_m row tiles; within a group the row
// tile varies fastest, so CTAs running at the same time share column tiles
// (the B operand) and a small set of row tiles (the A operand) in L2.
__device__ __forceinline__ void tile_coords(const GemmParams& p, int t, int& mt, int& nt) {
  const int per_group = p.group_m * p.n_nt;
  const int g = t / per_group;
  const int first = g * p.group_m;
  const int gm = min(p.group_m, p.n_mt - first);
  const int r = t - g * per_group;
  mt = first + r % gm;
  nt = r / gm;
}

// One accumulator row (this thread's TMEM lane, 256 columns from tbase) to
// memory.  Every lane runs every tcgen05.ld (they are warp-collective);
// only the stores depend on the row being inside the output.  N is a
// multiple of 64, so each 32-column chunk is wholly inside or outside it,
// the same for the whole warp.
template <int EPI>
__device__ __forceinline__ void epilogue_tile(const GemmParams& p, uint32_t tbase, int row,
                                              bool row_ok, int n0, int nt) {
  if constexpr (EPI == EPI_LOGITS) {
    const int tgt = row_ok ? __ldg(p.target + row) : -1;
    float m_run = -INFINITY, l_run = 0.f, zt = 0.f;
    bool has_t = false;
    float* zrow = p.z + static_cast<int64_t>(row) * p.ldz;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float v[32];
      tmem_ld32(tbase + c, v);
      const int col0 = n0 + c;
      if (col0 >= p.N) continue;
      if (row_ok) {
        float4* dst = reinterpret_cast<float4*>(zrow + col0);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
      }
      float cm = v[0];
#pragma unroll
      for (int j = 1; j < 32; ++j) cm = fmaxf(cm, v[j]);
      const float mn = fmaxf(m_run, cm);
      const float mn2 = mn * kLog2e;
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) acc += ex2_approx(fmaf(v[j], kLog2e, -mn2));
      l_run = fmaf(l_run, ex2_approx((m_run - mn) * kLog2e), acc);  // 0 * 0 while m_run = -inf
      m_run = mn;
      if (tgt >= col0 && tgt < col0 + 32) {
#pragma unroll
        for (int j = 0; j < 32; ++j) zt = (col0 + j == tgt) ? v[j] : zt;
        has_t = true;
      }
    }
    if (row_ok) {
      p.part[static_cast<int64_t>(row) * p.n_nt + nt] = make_float2(m_run, l_run);
      if (has_t) p.zt[row] = zt;
    }
  } else if constexpr (EPI == EPI_BF16) {
    __nv_bfloat16* orow = static_cast<__nv_bfloat16*>(p.out) + static_cast<int64_t>(row) * p.ld_out;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float v[32];
      tmem_ld32(tbase + c, v);
      const int col0 = n0 + c;
      if (col0 >= p.N || !row_ok) continue;
      uint4* dst = reinterpret_cast<uint4*>(orow + col0);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        dst[j] = make_uint4(pack_bf16x2(v[8 * j], v[8 * j + 1]), pack_bf16x2(v[8 * j + 2], v[8 * j + 3]),
                            pack_bf16x2(v[8 * j + 4], v[8 * j + 5]),
                            pack_bf16x2(v[8 * j + 6], v[8 * j + 7]));
    }
  } else {
    float* orow = static_cast<float*>(p.out) + static_cast<int64_t>(row) * p.ld_out;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      float v[32];
      tmem_ld32(tbase + c, v);
      const int col0 = n0 + c;
      if (col0 >= p.N || !row_ok) continue;
      float4* dst = reinterpret_cast<float4*>(orow + col0);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        float4 o = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
        if (p.accumulate) {
          const float4 e = dst[j];
          o.x += e.x;
          o.y += e.y;
          o.z += e.z;
          o.w += e.w;
        }
        dst[j] = o;
      }
    }
  }
}

// A: M x K operand, K-major ([M][K] in memory, box 64 x 128) or MN-major
// ([K][M], two 64 x 64 boxes).  B: N x K, K-major (box 64 x 256) or
// MN-major ([K][N], four 64 x 64 boxes).  MN-major tiles sit in shared memory
// as 64-element chunks of 64 K rows (8 KB apart: the descriptor's leading
// byte offset); K-major tiles as rows of 64 K elements (8-row atoms 1 KB
// apart: the stride byte offset).
template <int EPI, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(kGemmThreads, 1)
    ce_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  if (smem_u32(smem) & 1023u) {
    if (threadIdx.x == 0) atomicExch(p.status, DEV_MISALIGNED);
    return;
  }
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kSmemBar);
  uint32_t* tmem_sh = reinterpret_cast<uint32_t*>(smem + kSmemMisc);
  int* abort_flag = reinterpret_cast<int*>(smem + kSmemMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nk = (p.K + BK - 1) / BK;

  if (threadIdx.x == 0) {
    for (int i = 0; i < G_COUNT; ++i) mbar_init(&bars[i], (i == G_ACC_EMPTY || i == G_ACC_EMPTY + 1) ? 4 : 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_sh, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_sh;

  if (warp == 0) {
    if (lane == 0) {
      // ===================== TMA producer
      prefetch_tmap(&tm_a);
      prefetch_tmap(&tm_b);
      int it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x) {
        int mt, nt;
        tile_coords(p, t, mt, nt);
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          if (it >= kStages) {
            ok = mbar_wait(&bars[G_EMPTY + s], ((it / kStages) + 1) & 1, p.status, abort_flag);
            if (!ok) break;
          }
          uint64_t* full = &bars[G_FULL + s];
          mbar_arrive_expect_tx(full, kABytes + kBBytes);
          uint8_t* a = smem + kSmemA + s * kABytes;
          uint8_t* b = smem + kSmemB + s * kBBytes;
          if (A_MN) {
            tma_load_2d(a, &tm_a, full, mt * BM, kb * BK);
            tma_load_2d(a + kChunkBytes, &tm_a, full, mt * BM + 64, kb * BK);
          } else {
            tma_load_2d(a, &tm_a, full, kb * BK, mt * BM);
          }
          if (B_MN) {
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_2d(b + j * kChunkBytes, &tm_b, full, nt * BN + 64 * j, kb * BK);
          } else {
            tma_load_2d(b, &tm_b, full, kb * BK, nt * BN);
          }
        }
      }
      if (!ok) {
        // drain: the loads of the last (up to kStages) issued steps
        for (int i = (it > kStages ? it - kStages : 0); i < it; ++i)
          mbar_wait(&bars[G_FULL + i % kStages], (i / kStages) & 1, nullptr, nullptr, kDrainNs);
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ===================== MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN, A_MN, B_MN);
      constexpr uint32_t a_step = A_MN ? 2048u : 32u;  // bytes per K = 16
      constexpr uint32_t b_step = B_MN ? 2048u : 32u;
      int it = 0, tc = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.n_tiles && ok; t += gridDim.x, ++tc) {
        const int buf = tc & 1;
        if (tc >= 2) {
          ok = mbar_wait(&bars[G_ACC_EMPTY + buf], ((tc >> 1) - 1) & 1, p.status, abort_flag);
          if (!ok) break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + buf * BN;
        for (int kb = 0; kb < nk; ++kb, ++it) {
          const int s = it % kStages;
          ok = mbar_wait(&bars[G_FULL + s], (it / kStages) & 1, p.status, abort_flag);
          if (!ok) break;
          tc_fence_after_sync();
          const uint64_t ad = sdesc_sw128(smem_u32(smem + kSmemA + s * kABytes),
                                          A_MN ? kChunkBytes : 16u, 1024);
          const uint64_t bd = sdesc_sw128(smem_u32(smem + kSmemB + s * kBBytes),
                                          B_MN ? kChunkBytes : 16u, 1024);
#pragma unroll
          for (int k = 0; k < BK / 16; ++k)
            umma_bf16_ss(d_tmem, sdesc_step(ad, k * a_step), sdesc_step(bd, k * b_step), idesc,
                         (kb > 0 || k > 0) ? 1u : 0u);
          umma_commit(&bars[G_EMPTY + s]);
        }
        if (!ok) break;
        umma_commit(&bars[G_ACC_FULL + buf]);
      }
      // every MMA issued by this thread completes before TMEM is released
      umma_commit(&bars[G_DRAIN]);
      mbar_wait(&bars[G_DRAIN], 0, nullptr, nullptr, kDrainNs);
    }
  } else if (warp >= 4) {
    // ===================== epilogue: warp 4 + w reads TMEM lanes 32w .. 32w + 31
    const int ew = warp - 4;
    const int r = ew * 32 + lane;
    int tc = 0;
    for (int t = blockIdx.x; t < p.n_tiles; t += gridDim.x, ++tc) {
      const int buf = tc & 1;
      if (!mbar_wait_warp(&bars[G_ACC_FULL + buf], (tc >> 1) & 1, p.status, abort_flag)) break;
      tc_fence_after_sync();
      int mt, nt;
      tile_coords(p, t, mt, nt);
      const int row = mt * BM + r;
      const bool row_ok = row < p.M;
      const int n0 = nt * BN;
      const uint32_t tbase = tmem + (static_cast<uint32_t>(ew * 32) << 16) + buf * BN;
      epilogue_tile<EPI>(p, tbase, row, row_ok, n0, nt);
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars[G_ACC_EMPTY + buf]);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

__device__ __forceinline__ float block_reduce(float v, bool is_max, float* red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = is_max ? fmaxf(v, w) : v + w;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  __syncthreads();  // red[] is reused by consecutive reductions
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = red[0];
#pragma unroll
  for (int w = 1; w < kRowThreads / 32; ++w) v = is_max ? fmaxf(v, red[w]) : v + red[w];
  return v;
}

// One row of the chunk per CTA: LSE from the per-tile (max, sum of exp)
// pairs, the loss, then g = s (exp(z - lse) - onehot) over the row's logits
// as bf16 (all zero for an ignored row).
__global__ void __launch_bounds__(kRowThreads)
    ce_row_kernel(const float* __restrict__ z, int64_t ldz, const float2* __restrict__ part, int n_vt,
                  const float* __restrict__ zt, const int32_t* __restrict__ target, int V, float scale,
                  float* __restrict__ loss, float* __restrict__ lse, __nv_bfloat16* __restrict__ g) {
  __shared__ float red[kRowThreads / 32];
  const int64_t row = blockIdx.x;
  const float2* pr = part + row * n_vt;
  float m = -INFINITY;
  for (int j = threadIdx.x; j < n_vt; j += kRowThreads) m = fmaxf(m, pr[j].x);
  m = block_reduce(m, true, red);
  float s = 0.f;
  for (int j = threadIdx.x; j < n_vt; j += kRowThreads) {
    const float2 q = pr[j];
    s = fmaf(q.y, ex2_approx((q.x - m) * kLog2e), s);
  }
  s = block_reduce(s, false, red);
  const float lse_r = m + logf(s);
  const int t = target[row];
  const bool valid = t >= 0 && t < V;
  if (threadIdx.x == 0) {
    lse[row] = lse_r;
    loss[row] = valid ? lse_r - zt[row] : 0.f;
  }
  const float sc = valid ? scale : 0.f;
  const float off = lse_r * kLog2e;
  const float4* zr = reinterpret_cast<const float4*>(z + row * ldz);
  uint2* gr = reinterpret_cast<uint2*>(g + row * static_cast<int64_t>(V));
  for (int i = threadIdx.x; i < V / 4; i += kRowThreads) {
    const float4 q = zr[i];
    const int v0 = 4 * i;
    const float e0 = sc * (ex2_approx(fmaf(q.x, kLog2e, -off)) - (v0 == t ? 1.f : 0.f));
    const float e1 = sc * (ex2_approx(fmaf(q.y, kLog2e, -off)) - (v0 + 1 == t ? 1.f : 0.f));
    const float e2 = sc * (ex2_approx(fmaf(q.z, kLog2e, -off)) - (v0 + 2 == t ? 1.f : 0.f));
    const float e3 = sc * (ex2_approx(fmaf(q.w, kLog2e, -off)) - (v0 + 3 == t ? 1.f : 0.f));
    gr[i] = make_uint2(pack_bf16x2(e0, e1), pack_bf16x2(e2, e3));
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return 0;
  return n;
}

template <int EPI, bool A_MN, bool B_MN>
cudaError_t launch_gemm(const CUtensorMap& a, const CUtensorMap& b, GemmParams p, int kind,
                        cudaStream_t stream) {
  auto kern = ce_gemm_kernel<EPI, A_MN, B_MN>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemTotal);
  if (e != cudaSuccess) return e;
  p.n_mt = (p.M + BM - 1) / BM;
  p.n_nt = (p.N + BN - 1) / BN;
  p.n_tiles = p.n_mt * p.n_nt;
  p.group_m = p.n_mt < 16 ? p.n_mt : 16;
  const int sms = sm_count();
  if (sms <= 0) return cudaErrorInvalidDevice;
  const int grid = p.n_tiles < sms ? p.n_tiles : sms;
  const int timed = timer_begin(kind, stream);
  kern<<<grid, kGemmThreads, kSmemTotal, stream>>>(a, b, p);
  e = cudaGetLastError();
  timer_end(timed, stream);
  return e;
}

struct CeLayout {
  int64_t chunk = 0, n_vt = 0;
  size_t z = 0, g = 0, part = 0, zt = 0, total = 0;
};

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

bool ce_valid(const csbp_ce_problem* p) {
  // rows x d_model below 2^39 elements (1 TiB of bf16 h): every row, element
  // and byte count below then stays inside int64 (tested by division)
  constexpr int64_t kMaxElems = int64_t(1) << 39;
  if (!p || p->rows < 1 || p->d_model < 64 || p->d_model > 65536 || p->d_model % 64 != 0 ||
      p->rows > (kMaxElems - 1) / p->d_model ||
      p->vocab < 64 || p->vocab > (1 << 24) || p->vocab % 64 != 0 || p->chunk_rows < 0 ||
      p->chunk_rows % BM != 0 || (p->head_grad != 0 && p->head_grad != 1) ||
      !std::isfinite(p->grad_scale))
    return false;
  return true;
}

CeLayout ce_layout(const csbp_ce_problem* p) {
  CeLayout l;
  const int64_t want = p->chunk_rows > 0 ? p->chunk_rows : kDefaultChunk;
  const int64_t rows_up = (p->rows + BM - 1) / BM * BM;
  l.chunk = want < rows_up ? want : rows_up;
  l.n_vt = (p->vocab + BN - 1) / BN;
  size_t off = 256;  // status word
  l.z = off;
  off += round256(static_cast<size_t>(l.chunk) * p->vocab * 4);
  l.g = off;
  off += round256(static_cast<size_t>(l.chunk) * p->vocab * 2);
  l.part = off;
  off += round256(static_cast<size_t>(l.chunk) * l.n_vt * 8);
  l.zt = off;
  off += round256(static_cast<size_t>(l.chunk) * 4);
  l.total = off;
  return l;
}

bool aligned16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

}  // namespace
}  // namespace csbp

using namespace csbp;

extern "C" size_t csbp_ce_workspace_bytes(const csbp_ce_problem* problem) {
  if (!ce_valid(problem)) return 0;
  return ce_layout(problem).total;
}

extern "C" csbp_status csbp_vocab_ce(const csbp_ce_problem* problem, const void* h, const void* w,
                                     const int32_t* target, float* loss, float* lse, void* dh,
                                     float* dw, void* workspace, size_t workspace_bytes,
                                     void* stream_) {
  if (!ce_valid(problem)) return CSBP_ERR_INVALID;
  const csbp_ce_problem& p = *problem;
  const void* ptrs[7] = {h, w, target, loss, lse, dh, workspace};
  for (const void* q : ptrs)
    if (!q || !aligned16(q)) return CSBP_ERR_INVALID;
  if (p.head_grad ? (!dw || !aligned16(dw)) : (dw != nullptr)) return CSBP_ERR_INVALID;
  const CeLayout lay = ce_layout(&p);
  if (workspace_bytes < lay.total) return CSBP_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int* status = reinterpret_cast<int*>(ws);
  float* z = reinterpret_cast<float*>(ws + lay.z);
  __nv_bfloat16* g = reinterpret_cast<__nv_bfloat16*>(ws + lay.g);
  float2* part = reinterpret_cast<float2*>(ws + lay.part);
  float* zt = reinterpret_cast<float*>(ws + lay.zt);
  const int64_t Dm = p.d_model, V = p.vocab;
  const uint8_t* hb = static_cast<const uint8_t*>(h);

  CUtensorMap m_w_k, m_w_mn;  // W as K-major B (logits) and MN-major B (dH)
  if (!encode_map_2d(&m_w_k, false, w, Dm, V, Dm * 2, 64, BN, true) ||
      !encode_map_2d(&m_w_mn, false, w, Dm, V, Dm * 2, 64, 64, true))
    return CSBP_ERR_CUDA;

  for (int64_t c0 = 0; c0 < p.rows; c0 += lay.chunk) {
    const int64_t rows = (p.rows - c0 < lay.chunk) ? p.rows - c0 : lay.chunk;
    const void* hc = hb + c0 * Dm * 2;
    CUtensorMap m_h_k, m_g_k, m_g_mn, m_h_mn;
    if (!encode_map_2d(&m_h_k, false, hc, Dm, rows, Dm * 2, 64, BM, true) ||
        !encode_map_2d(&m_g_k, false, g, V, rows, V * 2, 64, BM, true) ||
        !encode_map_2d(&m_g_mn, false, g, V, rows, V * 2, 64, 64, true) ||
        !encode_map_2d(&m_h_mn, false, hc, Dm, rows, Dm * 2, 64, 64, true))
      return CSBP_ERR_CUDA;

    GemmParams gp{};
    gp.status = status;
    // 1. logits, per-tile softmax partials, target logits
    gp.M = static_cast<int32_t>(rows);
    gp.N = static_cast<int32_t>(V);
    gp.K = static_cast<int32_t>(Dm);
    gp.z = z;
    gp.ldz = V;
    gp.part = part;
    gp.zt = zt;
    gp.target = target + c0;
    if (launch_gemm<EPI_LOGITS, false, false>(m_h_k, m_w_k, gp, 2, stream) != cudaSuccess)
      return CSBP_ERR_CUDA;
    // 2. LSE, loss, g
    {
      const int timed = timer_begin(3, stream);
      ce_row_kernel<<<static_cast<unsigned>(rows), kRowThreads, 0, stream>>>(
          z, V, part, static_cast<int>(lay.n_vt), zt, target + c0, static_cast<int>(V),
          p.grad_scale, loss + c0, lse + c0, g);
      const cudaError_t e = cudaGetLastError();
      timer_end(timed, stream);
      if (e != cudaSuccess) return CSBP_ERR_CUDA;
    }
    // 3. dH = g W
    GemmParams hp{};
    hp.status = status;
    hp.M = static_cast<int32_t>(rows);
    hp.N = static_cast<int32_t>(Dm);
    hp.K = static_cast<int32_t>(V);
    hp.out = static_cast<uint8_t*>(dh) + c0 * Dm * 2;
    hp.ld_out = Dm;
    if (launch_gemm<EPI_BF16, false, true>(m_g_k, m_w_mn, hp, 4, stream) != cudaSuccess)
      return CSBP_ERR_CUDA;
    // 4. dW (+)= g^T H_c
    if (p.head_grad) {
      GemmParams wp{};
      wp.status = status;
      wp.M = static_cast<int32_t>(V);
      wp.N = static_cast<int32_t>(Dm);
      wp.K = static_cast<int32_t>(rows);
      wp.out = dw;
      wp.ld_out = Dm;
      wp.accumulate = c0 > 0 ? 1 : 0;
      if (launch_gemm<EPI_F32, true, true>(m_g_mn, m_h_mn, wp, 5, stream) != cudaSuccess)
        return CSBP_ERR_CUDA;
    }
  }
  return CSBP_OK;
}
