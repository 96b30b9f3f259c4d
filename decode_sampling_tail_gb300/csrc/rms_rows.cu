// Final RMSNorm of the tail ("GPT-OSS Tail Chunked Megakernel Kernel API
// Reference", parameters `hidden_states`, `gamma`, `eps`, `hidden_actual`,
// `zero_interleaved_pad`, `deferred_rms`).
//
// One CTA per batch row:
//   1. widen the row to fp32 (exact: every bf16 and fp16 value is an fp32 value);
//   2. ss = sum of x^2 over the active lanes (all H lanes when the pads are
//      zero, else lanes [0, H_u)); rstd = 1 / sqrt(ss / H_u + eps);
//   3. a = x * gamma (deferred: rstd is applied to the GEMM output) or
//      a = (x * rstd) * gamma (legacy form feeding the GEMM);
//   4. split a = hi + lo into two bf16 values (hi = bf16(a), lo = bf16(a - hi))
//      so the bf16 tensor-core GEMM keeps about 16 significant bits of the
//      activation, and store both in mma.sync m16n8k16 A-fragment order:
//      m-tile = 8 batch rows, fragment rows 0-7 are their hi parts, rows 8-15
//      their lo parts.
// Rows in [B, B_pad) are written as zeros so the last m-tile is complete.
#include "common.cuh"
#include "internal.h"
#include "moe.cuh"
#include "tc_internal.h"

namespace tail {

namespace {

constexpr int RMS_THREADS = 256;

template <int DT>
__device__ __forceinline__ float load_widen(const void* p, int64_t i) {
  if constexpr (DT == 0) {
    return static_cast<const float*>(p)[i];
  } else if constexpr (DT == 1) {
    return __half2float(static_cast<const __half*>(p)[i]);
  } else {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  }
}

__device__ __forceinline__ uint32_t bf16_bits(float v) {
  return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(v)));
}

// Word offset of the (hi or lo) register pair holding k-columns (kk, kk+1) of
// batch row g of m-tile mt in k-step ks.  kk is even.
__device__ __forceinline__ int64_t pack_word(int ks, int mt, int n_mt, int g, int kk, int lo) {
  const int lane = g * 4 + ((kk & 7) >> 1);
  const int reg = (kk < 8 ? 0 : 2) + lo;
  return ((static_cast<int64_t>(ks) * n_mt + mt) * 32 + lane) * 4 + reg;
}

template <int DT>
__global__ void __launch_bounds__(RMS_THREADS) rms_pack_kernel(RmsArgs a) {
  pdl_wait();  // scratch is reused across steps: wait for the previous step to finish with it
  pdl_launch_dependents();
  __shared__ float red[RMS_THREADS / 32];
  __shared__ float s_rstd;
  const int b = blockIdx.x;
  const int mt = b / MTILE_ROWS, g = b % MTILE_ROWS;
  const int H = a.H;

  if (b >= a.B) {  // padding rows of the last m-tile
    for (int h2 = 2 * threadIdx.x; h2 < H; h2 += 2 * RMS_THREADS) {
      a.apack[pack_word(h2 / KSTEP, mt, a.mt, g, h2 % KSTEP, 0)] = 0u;
      a.apack[pack_word(h2 / KSTEP, mt, a.mt, g, h2 % KSTEP, 1)] = 0u;
    }
    if (threadIdx.x == 0) a.row_scale[b] = 0.f;
    return;
  }

  const int64_t row = static_cast<int64_t>(b) * H;
  const int active_end = a.zero_pad ? H : a.Hu;
  float ss = 0.f;
  for (int h = threadIdx.x; h < active_end; h += RMS_THREADS) {
    const float v = load_widen<DT>(a.hidden, row + h);
    ss = fmaf(v, v, ss);
  }
  // fixed-order reduction: xor butterfly in each warp, then warps in order
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < RMS_THREADS / 32; ++w) t += red[w];
    s_rstd = 1.0f / sqrtf(t / static_cast<float>(a.Hu) + a.eps);
  }
  __syncthreads();
  const float rstd = s_rstd;
  const float pre = a.deferred ? 1.0f : rstd;

  for (int h2 = 2 * threadIdx.x; h2 < H; h2 += 2 * RMS_THREADS) {
    float v[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int h = h2 + j;
      if (h < active_end) {
        const float x = load_widen<DT>(a.hidden, row + h);
        v[j] = (x * pre) * a.gamma[h];
      } else {
        v[j] = 0.f;
      }
    }
    uint32_t hi[2], lo[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      hi[j] = bf16_bits(v[j]);
      const float hif = __uint_as_float(hi[j] << 16);
      lo[j] = bf16_bits(v[j] - hif);
    }
    const int ks = h2 / KSTEP, kk = h2 % KSTEP;
    a.apack[pack_word(ks, mt, a.mt, g, kk, 0)] = hi[0] | (hi[1] << 16);
    a.apack[pack_word(ks, mt, a.mt, g, kk, 1)] = lo[0] | (lo[1] << 16);
  }
  if (threadIdx.x == 0) a.row_scale[b] = a.deferred ? rstd : 1.0f;
}

// The same RMSNorm for the tensor-core path: the hi and lo parts of row b go
// to their rows of the activation image (tc_internal.h: the tensor-core
// kernel's shared-memory stages, 128-byte swizzle included), k-columns up to
// the last k-block's end (zeros past H).  A thread takes groups of 8
// consecutive columns (one 16-byte load of 16-bit elements, two of fp32; one
// 16-byte store each of hi and lo): Σx² runs group by group, then over the
// warps in order, so rstd is deterministic and the same for every input type.
// MOE: the row is first formed by the producer step (moe.cuh) from the
// residual and the expert slots -- h, kept in shared memory as bf16 and
// written to the caller's buffer when one is given -- and the RMSNorm runs on
// it in the same order as on a bf16 input.
template <int DT>
__device__ __forceinline__ void load8_widen(const void* p, int64_t i, float (&x)[8]) {
  if constexpr (DT == 0) {
    const float4 u = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i);
    const float4 w = *reinterpret_cast<const float4*>(static_cast<const float*>(p) + i + 4);
    x[0] = u.x; x[1] = u.y; x[2] = u.z; x[3] = u.w;
    x[4] = w.x; x[5] = w.y; x[6] = w.z; x[7] = w.w;
  } else {
    const uint4 u = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p) + i);
    const uint32_t q[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const uint16_t e0 = static_cast<uint16_t>(q[j] & 0xFFFFu), e1 = static_cast<uint16_t>(q[j] >> 16);
      if constexpr (DT == 1) {
        x[2 * j] = __half2float(__ushort_as_half(e0));
        x[2 * j + 1] = __half2float(__ushort_as_half(e1));
      } else {
        x[2 * j] = __uint_as_float(static_cast<uint32_t>(e0) << 16);
        x[2 * j + 1] = __uint_as_float(static_cast<uint32_t>(e1) << 16);
      }
    }
  }
}

template <int DT, bool MOE>
__global__ void __launch_bounds__(RMS_THREADS) rms_split_kernel(SplitArgs a) {
  pdl_wait();  // the activation buffer is reused across steps
  pdl_launch_dependents();
  __shared__ float red[RMS_THREADS / 32];
  __shared__ float s_rstd;
  extern __shared__ uint16_t s_h[];  // MOE: the row's h
  const int b = blockIdx.x;
  const int H = a.H;  // a multiple of 16
  const int64_t row = static_cast<int64_t>(b) * H;
  const int active_end = a.zero_pad ? H : a.Hu;
  auto group = [&](int h0, float (&x)[8]) {  // columns h0 .. h0 + 7 of the row
    if constexpr (MOE) {
#pragma unroll
      for (int j = 0; j < 8; ++j) x[j] = __uint_as_float(static_cast<uint32_t>(s_h[h0 + j]) << 16);
    } else {
      load8_widen<DT>(a.hidden, row + h0, x);
    }
  };
  float ss = 0.f;
  for (int g = threadIdx.x; g < H / 8; g += RMS_THREADS) {
    const int h0 = 8 * g;
    float x[8];
    if constexpr (MOE) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t hb = moe_lane_h(a.moe, b, H, h0 + j);
        s_h[h0 + j] = static_cast<uint16_t>(hb);
        if (a.moe.h_out) a.moe.h_out[row + h0 + j] = static_cast<uint16_t>(hb);
        x[j] = __uint_as_float(hb << 16);
      }
    } else {
      group(h0, x);
    }
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (h0 + j < active_end) ss = fmaf(x[j], x[j], ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < RMS_THREADS / 32; ++w) t += red[w];
    s_rstd = 1.0f / sqrtf(t / static_cast<float>(a.Hu) + a.eps);
  }
  __syncthreads();
  const float rstd = s_rstd;
  const float pre = a.deferred ? 1.0f : rstd;
  const int kblocks = (H + TC_KB - 1) / TC_KB;
  for (int g = threadIdx.x; g < kblocks * (TC_KB / 8); g += RMS_THREADS) {
    const int h0 = 8 * g;
    float x[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.f;
    if (h0 < H) group(h0, x);
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int j = 0; j < 8; j += 2) {
      uint32_t hb[2], lb[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int h = h0 + j + u;
        const float v = h < active_end ? (x[j + u] * pre) * a.gamma[h] : 0.f;
        hb[u] = bf16_bits(v);
        lb[u] = bf16_bits(v - __uint_as_float(hb[u] << 16));
      }
      hi[j / 2] = hb[0] | (hb[1] << 16);
      lo[j / 2] = lb[0] | (lb[1] << 16);
    }
    *reinterpret_cast<uint4*>(a.act_img + tc_act_image_offset(a.stacked, kblocks, b, 0, h0)) =
        make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(a.act_img + tc_act_image_offset(a.stacked, kblocks, b, 1, h0)) =
        make_uint4(lo[0], lo[1], lo[2], lo[3]);
  }
  if (threadIdx.x == 0) a.row_scale[b] = a.deferred ? rstd : 1.0f;
}

}  // namespace

cudaError_t launch_split(const SplitArgs& a, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B);
  cfg.blockDim = dim3(RMS_THREADS);
  cfg.dynamicSmemBytes = a.use_moe ? static_cast<size_t>(a.H) * 2 : 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (a.use_moe) {
    if (a.H > SPLIT_MOE_MAX_H) return cudaErrorInvalidValue;
    return cudaLaunchKernelEx(&cfg, rms_split_kernel<2, true>, a);
  }
  switch (a.dtype) {
    case 0: return cudaLaunchKernelEx(&cfg, rms_split_kernel<0, false>, a);
    case 1: return cudaLaunchKernelEx(&cfg, rms_split_kernel<1, false>, a);
    case 2: return cudaLaunchKernelEx(&cfg, rms_split_kernel<2, false>, a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_rms_pack(const RmsArgs& a, cudaStream_t stream, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.B_pad);
  cfg.blockDim = dim3(RMS_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  switch (a.dtype) {
    case 0: return cudaLaunchKernelEx(&cfg, rms_pack_kernel<0>, a);
    case 1: return cudaLaunchKernelEx(&cfg, rms_pack_kernel<1>, a);
    case 2: return cudaLaunchKernelEx(&cfg, rms_pack_kernel<2>, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tail
