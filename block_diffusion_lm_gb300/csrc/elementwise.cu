// Bandwidth-bound kernels of the attention path:
//  * exact log-sum-exp merge of partial attentions ("CSBP 完全拆解" blog,
//    section "在线 softmax 合并：为什么分两段算仍是同一个注意力": m = max z_s,
//    w_s = exp(z_s - m), O = sum w_s O_s / sum w_s, z = m + log sum w_s, fp32
//    until the final bf16 rounding of O);
//  * backward preprocessing D_i = sum_c dO_ic O_ic (fp32) fused with zeroing
//    the fp32 dQ accumulator rows;
//  * dQ accumulator (fp32) -> scaled bf16;
//  * fill of the partial-LSE buffer with -inf (parts that read no key);
//  * fp8 E4M3 inputs times a per-tensor scale -> bf16 (inputs kept in fp8).
// Grids are sized as a multiple of the SM count and walk their range with a
// grid stride; every access is 16-byte vectorised.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "csbp_internal.h"

namespace csbp {

namespace {

// One thread per 4 consecutive head-dim elements of one (row, head).
__global__ void __launch_bounds__(256) lse_merge_kernel(MergeArgs a, int n_parts, int64_t rows,
                                                        int Hq, int d, __nv_bfloat16* o_out,
                                                        float* z_out) {
  const int d4 = d >> 2;
  const int64_t total = rows * Hq * d4;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t rh = idx / d4;
    const int c4 = static_cast<int>(idx - rh * d4);
    const int64_t row = rh / Hq;
    const int h = static_cast<int>(rh - row * Hq);
    const int64_t zi = static_cast<int64_t>(h) * rows + row;
    float m = -INFINITY;
    for (int s = 0; s < n_parts; ++s) m = fmaxf(m, __ldg(a.z[s] + zi));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (m != -INFINITY) {
      for (int s = 0; s < n_parts; ++s) {
        const float zs = __ldg(a.z[s] + zi);
        if (zs == -INFINITY) continue;  // the part read no key: weight 0
        const float w = expf(zs - m);
        const float4 v = __ldg(reinterpret_cast<const float4*>(a.o[s] + rh * d) + c4);
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
        wsum += w;
      }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(o_out + rh * d + c4 * 4) = packed;
    if (c4 == 0) z_out[zi] = (wsum > 0.f) ? m + logf(wsum) : -INFINITY;
  }
}

// D[qs][b][h][pos] = sum_c dO * O over one (row, head); G8 = d/8 threads per
// row each holding 8 bf16 of both operands.  Also zeroes that row's fp32 dQ
// accumulator.
template <int D>
__global__ void __launch_bounds__(256) bwd_pre_kernel(const __nv_bfloat16* o, const __nv_bfloat16* dO,
                                                      float* Dsum, float* dq_acc, int64_t rows,
                                                      int Hq, int L) {
  constexpr int kG = D / 8;  // threads per (row, head)
  const int64_t total = rows * Hq * kG;
  for (int64_t idx = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; idx < total;
       idx += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t rh = idx / kG;
    const int g = static_cast<int>(idx - rh * kG);
    const uint4 ov = __ldg(reinterpret_cast<const uint4*>(o + rh * D) + g);
    const uint4 dv = __ldg(reinterpret_cast<const uint4*>(dO + rh * D) + g);
    const __nv_bfloat162* op = reinterpret_cast<const __nv_bfloat162*>(&ov);
    const __nv_bfloat162* dp = reinterpret_cast<const __nv_bfloat162*>(&dv);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = __bfloat1622float2(op[k]);
      const float2 b = __bfloat1622float2(dp[k]);
      s += a.x * b.x + a.y * b.y;
    }
    // groups of kG lanes are aligned and enter/leave the loop together
    const unsigned active = __activemask();
#pragma unroll
    for (int off = kG / 2; off > 0; off >>= 1) s += __shfl_xor_sync(active, s, off, kG);
    float4* acc = reinterpret_cast<float4*>(dq_acc + rh * D) + 2 * g;
    acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
    acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    if (g == 0) {
      // rh = (b * L + pos) * Hq + h  ->  Dsum[b][h][pos]
      const int64_t bp = rh / Hq;
      const int h = static_cast<int>(rh - bp * Hq);
      const int64_t b = bp / L;
      const int64_t pos = bp - b * L;
      Dsum[(b * Hq + h) * L + pos] = s;
    }
  }
}

__global__ void __launch_bounds__(256) dq_convert_kernel(const float* acc, __nv_bfloat16* dq,
                                                         int64_t n8, float scale) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i);
    const float4 b = __ldg(reinterpret_cast<const float4*>(acc) + 2 * i + 1);
    __nv_bfloat162 v0 = __floats2bfloat162_rn(a.x * scale, a.y * scale);
    __nv_bfloat162 v1 = __floats2bfloat162_rn(a.z * scale, a.w * scale);
    __nv_bfloat162 v2 = __floats2bfloat162_rn(b.x * scale, b.y * scale);
    __nv_bfloat162 v3 = __floats2bfloat162_rn(b.z * scale, b.w * scale);
    uint4 u;
    u.x = *reinterpret_cast<uint32_t*>(&v0);
    u.y = *reinterpret_cast<uint32_t*>(&v1);
    u.z = *reinterpret_cast<uint32_t*>(&v2);
    u.w = *reinterpret_cast<uint32_t*>(&v3);
    reinterpret_cast<uint4*>(dq)[i] = u;
  }
}

// Two E4M3 values (low byte first) -> two fp32, through the hardware
// conversion to f16x2, which is exact: every E4M3 value is an f16 value.
__device__ __forceinline__ float2 e4m3x2_to_float2(uint32_t two) {
  uint32_t h2;
  const uint16_t v = static_cast<uint16_t>(two & 0xffffu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  __half2 h;
  *reinterpret_cast<uint32_t*>(&h) = h2;
  return __half22float2(h);
}

__device__ __forceinline__ uint32_t bf16x2_bits(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

// out[i] = bf16_rn(scale * e4m3(in[i])): 16 inputs per thread (one 16-byte
// load, two 16-byte stores); the last n % 16 elements one per thread.
__global__ void __launch_bounds__(256) e4m3_to_bf16_kernel(const uint8_t* in, __nv_bfloat16* out,
                                                           int64_t n, float scale) {
  const int64_t n16 = n >> 4;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n16;
       i += stride) {
    const uint4 v = __ldg(reinterpret_cast<const uint4*>(in) + i);
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = e4m3x2_to_float2(w[k]);
      const float2 b = e4m3x2_to_float2(w[k] >> 16);
      o[2 * k] = bf16x2_bits(a.x * scale, a.y * scale);
      o[2 * k + 1] = bf16x2_bits(b.x * scale, b.y * scale);
    }
    uint4* dst = reinterpret_cast<uint4*>(out) + 2 * i;
    dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
  for (int64_t i = (n16 << 4) + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x;
       i < n; i += stride)
    out[i] = __float2bfloat16_rn(e4m3x2_to_float2(in[i]).x * scale);
}

__global__ void __launch_bounds__(256) fill_kernel(float* x, int64_t n, float v) {
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x)
    x[i] = v;
}

int grid_for(int64_t work_items) {
  // SM count of the device in use at the first call (a thread-safe static);
  // 152, the GB300's count, if the query fails
  static const int sms = [] {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
      return 152;
    return n;
  }();
  const int64_t blocks = (work_items + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sms) * 8;  // 8 resident 256-thread CTAs per SM
  return static_cast<int>(blocks < cap ? (blocks > 0 ? blocks : 1) : cap);
}

}  // namespace

cudaError_t launch_lse_merge(const MergeArgs& a, int n_parts, int64_t rows, int Hq, int d,
                             void* o_out, float* z_out, cudaStream_t stream) {
  const int64_t total = rows * Hq * (d / 4);
  lse_merge_kernel<<<grid_for(total), 256, 0, stream>>>(a, n_parts, rows, Hq, d,
                                                        static_cast<__nv_bfloat16*>(o_out), z_out);
  return cudaGetLastError();
}

cudaError_t launch_bwd_pre(int d, const void* o, const void* dO, float* Dsum, float* dq_acc,
                           int64_t rows, int Hq, int L, cudaStream_t stream) {
  const int64_t total = rows * Hq * (d / 8);
  if (d == 128)
    bwd_pre_kernel<128><<<grid_for(total), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), Dsum, dq_acc,
        rows, Hq, L);
  else
    bwd_pre_kernel<64><<<grid_for(total), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), Dsum, dq_acc,
        rows, Hq, L);
  return cudaGetLastError();
}

cudaError_t launch_dq_convert(const float* acc, void* dq, int64_t n_elems, float scale,
                              cudaStream_t stream) {
  const int64_t n8 = n_elems / 8;
  dq_convert_kernel<<<grid_for(n8), 256, 0, stream>>>(acc, static_cast<__nv_bfloat16*>(dq), n8,
                                                      scale);
  return cudaGetLastError();
}

cudaError_t launch_e4m3_to_bf16(const void* in, void* out, int64_t n, float scale,
                                cudaStream_t stream) {
  const int64_t work = (n >> 4) > 0 ? (n >> 4) : 1;
  e4m3_to_bf16_kernel<<<grid_for(work), 256, 0, stream>>>(
      static_cast<const uint8_t*>(in), static_cast<__nv_bfloat16*>(out), n, scale);
  return cudaGetLastError();
}

cudaError_t launch_fill(float* x, int64_t n, float v, cudaStream_t stream) {
  fill_kernel<<<grid_for(n), 256, 0, stream>>>(x, n, v);
  return cudaGetLastError();
}

}  // namespace csbp
