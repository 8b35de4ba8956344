// The block around the scan, as in the mamba_split_conv1d_scan_combined call
// of the repro script on state-spaces/mamba issue #647 (the input projection
// split into z | xBC | dt, a causal depthwise conv1d with bias and SiLU over
// xBC, the scan, and an RMSNorm over groups of channels of the gated scan
// output, norm_before_gate=False):
//   causal_conv1d   out[b,t,c] = act(bias[c] + sum_k w[c,k] x[b, t-W+1+k, c])
//                   (taps before the sequence start, or in an earlier
//                   document of seq_idx, are zero)
//   group_rmsnorm   y[b,t,c] *= weight[c] / sqrt(mean_{c' in group(c)} y^2 + eps)
// Both are HBM-bound CUDA-core kernels: every input element is read once
// (the conv keeps its W-1 previous inputs in registers while it walks a run
// of tokens; the norm's second pass over a row hits L1/L2).
#include <math.h>
#include <stdio.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"

namespace ssd {
namespace block {

constexpr int kConvMaxW = 8;   // filter widths 1..8 (Mamba uses 4)
constexpr int kConvRun = 64;   // tokens per thread: the W-1 halo is re-read once per run
constexpr int kVec = 8;        // channels per thread (one 16-byte bf16 or two fp32 vectors)

__device__ __forceinline__ float silu_f(float v) { return v / (1.f + __expf(-v)); }

template <typename T>
__device__ __forceinline__ void load8(const T* p, float (&v)[kVec]) {
#pragma unroll
  for (int i = 0; i < kVec; ++i) v[i] = to_f(p[i]);
}
template <>
__device__ __forceinline__ void load8<__nv_bfloat16>(const __nv_bfloat16* p, float (&v)[kVec]) {
  const uint4 w = *reinterpret_cast<const uint4*>(p);
  const uint32_t u[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(u[i] << 16);
    v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void load8<float>(const float* p, float (&v)[kVec]) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

template <typename T>
__device__ __forceinline__ void store8(T* p, const float (&v)[kVec]);
template <>
__device__ __forceinline__ void store8<__nv_bfloat16>(__nv_bfloat16* p, const float (&v)[kVec]) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
    u[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  *reinterpret_cast<uint4*>(p) = make_uint4(u[0], u[1], u[2], u[3]);
}
template <>
__device__ __forceinline__ void store8<float>(float* p, const float (&v)[kVec]) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// The raw bits of one token's kVec channels (16 bytes of bf16 or 32 of
// fp32), held in registers ahead of their use, and their values.
struct Raw8 {
  uint4 a, b;
};
template <typename T>
__device__ __forceinline__ void raw_load(const T* p, Raw8& r) {
  r.a = *reinterpret_cast<const uint4*>(p);
  if constexpr (sizeof(T) == 4) r.b = *reinterpret_cast<const uint4*>(p + 4);
}
template <typename T>
__device__ __forceinline__ void raw_values(const Raw8& r, float (&v)[kVec]) {
  if constexpr (sizeof(T) == 2) {
    const uint32_t u[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(u[i] << 16);
      v[2 * i + 1] = __uint_as_float(u[i] & 0xFFFF0000u);
    }
  } else {
    const uint32_t u[8] = {r.a.x, r.a.y, r.a.z, r.a.w, r.b.x, r.b.y, r.b.z, r.b.w};
#pragma unroll
    for (int i = 0; i < kVec; ++i) v[i] = __uint_as_float(u[i]);
  }
}

// grid (ceil(C/8 / 128), ceil(L / kConvRun), B), 128 threads: thread ->
// 8 consecutive channels, a run of kConvRun tokens, with the filter and the
// last W inputs in registers.  A warp's loads of one token are 32 x 16
// contiguous bytes; each thread keeps the next two tokens' loads in flight
// (as raw bits, converted when used), since with the filter in registers
// few warps fit on an SM and one load each would leave HBM latency exposed.
template <typename T, int W>
__global__ void __launch_bounds__(128)
    causal_conv1d_kernel(const T* __restrict__ x, TokStride sx, const float* __restrict__ w,
                         const float* __restrict__ bias, const int32_t* __restrict__ seq_idx,
                         int64_t L, int C, int silu, T* __restrict__ out) {
  const int cg = blockIdx.x * blockDim.x + threadIdx.x;
  if (cg * kVec >= C) return;
  const int c0 = cg * kVec;
  const int b = blockIdx.z;
  const int64_t t0 = (int64_t)blockIdx.y * kConvRun;
  const int64_t t1 = t0 + kConvRun < L ? t0 + kConvRun : L;
  float wt[W][kVec], bv[kVec];
#pragma unroll
  for (int i = 0; i < kVec; ++i) {
    bv[i] = bias ? bias[c0 + i] : 0.f;
#pragma unroll
    for (int k = 0; k < W; ++k) wt[k][i] = w[(c0 + i) * W + k];
  }
  // win[k] = input at token t - (W-1) + k (tap k); the W-1 before t0 first;
  // taps before the sequence start are zero
  float win[W][kVec];
  int sq_win[W];
  const int32_t* sq = seq_idx ? seq_idx + (int64_t)b * L : nullptr;
#pragma unroll
  for (int k = 0; k < W - 1; ++k) {
    const int64_t t = t0 - (W - 1) + k;
#pragma unroll
    for (int i = 0; i < kVec; ++i) win[k][i] = 0.f;
    sq_win[k] = -1;
    if (t >= 0) {
      load8(x + toff(sx, b, t) + c0, win[k]);
      sq_win[k] = sq ? sq[t] : 0;
    }
  }
  Raw8 ra, rb;   // tokens t and t + 1, loaded ahead
  if (t0 < t1) raw_load(x + toff(sx, b, t0) + c0, ra);
  if (t0 + 1 < t1) raw_load(x + toff(sx, b, t0 + 1) + c0, rb);
  auto step = [&](int64_t t, Raw8& r) {
    raw_values<T>(r, win[W - 1]);
    if (t + 2 < t1) raw_load(x + toff(sx, b, t + 2) + c0, r);   // this slot's next token
    const int sq_t = sq ? sq[t] : 0;
    sq_win[W - 1] = sq_t;
    float acc[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) acc[i] = bv[i];
#pragma unroll
    for (int k = 0; k < W; ++k) {
      if (sq_win[k] == sq_t) {   // taps in an earlier document are zero
#pragma unroll
        for (int i = 0; i < kVec; ++i) acc[i] = fmaf(wt[k][i], win[k][i], acc[i]);
      }
    }
    if (silu) {
#pragma unroll
      for (int i = 0; i < kVec; ++i) acc[i] = silu_f(acc[i]);
    }
    store8(out + ((int64_t)b * L + t) * C + c0, acc);
#pragma unroll
    for (int k = 0; k < W - 1; ++k) {
      sq_win[k] = sq_win[k + 1];
#pragma unroll
      for (int i = 0; i < kVec; ++i) win[k][i] = win[k + 1][i];
    }
  };
  for (int64_t t = t0; t < t1; t += 2) {   // two tokens a turn: the slots alternate
    step(t, ra);
    if (t + 1 < t1) step(t + 1, rb);
  }
}

template <typename T>
cudaError_t launch_conv(const T* x, TokStride sx, const float* w, const float* bias,
                        const int32_t* seq_idx, int64_t B, int64_t L, int C, int W, int silu,
                        T* out, cudaStream_t st) {
  const int64_t nrun = (L + kConvRun - 1) / kConvRun;
  dim3 grid((unsigned)((C / kVec + 127) / 128), (unsigned)nrun, (unsigned)B);
  switch (W) {
#define SSD_CONV_W(n)                                                                         \
  case n:                                                                                     \
    causal_conv1d_kernel<T, n><<<grid, 128, 0, st>>>(x, sx, w, bias, seq_idx, L, C, silu, out); \
    break;
    SSD_CONV_W(1) SSD_CONV_W(2) SSD_CONV_W(3) SSD_CONV_W(4)
    SSD_CONV_W(5) SSD_CONV_W(6) SSD_CONV_W(7) SSD_CONV_W(8)
#undef SSD_CONV_W
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// One warp per (token, group): the sum of squares over the group's
// channels, then the scaled values written back in place.
template <typename T>
__global__ void __launch_bounds__(256)
    group_rmsnorm_kernel(T* __restrict__ y, const float* __restrict__ weight, float eps,
                         int64_t rows, int dim, int gs) {
  const int lane = threadIdx.x & 31;
  const int64_t wid = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int ng = dim / gs;
  if (wid >= rows * ng) return;
  const int64_t row = wid / ng;
  const int g = (int)(wid % ng);
  T* base = y + row * dim + (int64_t)g * gs;
  float ss = 0.f;
  for (int c = lane * kVec; c < gs; c += 32 * kVec) {
    float v[kVec];
    load8(base + c, v);
#pragma unroll
    for (int i = 0; i < kVec; ++i) ss = fmaf(v[i], v[i], ss);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  const float r = rsqrtf(ss / (float)gs + eps);
  for (int c = lane * kVec; c < gs; c += 32 * kVec) {
    float v[kVec];
    load8(base + c, v);
#pragma unroll
    for (int i = 0; i < kVec; ++i) v[i] = v[i] * r * weight[g * gs + c + i];
    store8(base + c, v);
  }
}

}  // namespace block
}  // namespace ssd

namespace {

int bad(int code, const char* msg) { return ssd::set_error(code, msg); }

bool al16(const void* p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" {

int ssd_causal_conv1d(const void* x, ssd_stride_t x_stride, const float* weight,
                      const float* bias, const int32_t* seq_idx, int64_t batch, int64_t seqlen,
                      int channels, int width, int silu, ssd_dtype_t dtype, void* out,
                      void* stream) {
  if (dtype != SSD_DTYPE_F32 && dtype != SSD_DTYPE_BF16) return bad(SSD_ERR_ARG, "unknown dtype");
  if (batch < 1 || seqlen < 1 || channels < 1 || batch > 65535)
    return bad(SSD_ERR_ARG, "batch (1..65535), seqlen and channels must be >= 1");
  if (channels % ssd::block::kVec != 0)
    return bad(SSD_ERR_UNSUPPORTED, "channels must be a multiple of 8");
  if (width < 1 || width > ssd::block::kConvMaxW)
    return bad(SSD_ERR_UNSUPPORTED, "width must be in [1, 8]");
  if (!x || !weight || !out) return bad(SSD_ERR_NULL, "x, weight and out are required");
  if (!al16(x) || !al16(out) || !al16(bias) || !al16(seq_idx) || ((uintptr_t)weight & 3u))
    return bad(SSD_ERR_ALIGN, "x, out, bias, seq_idx must be 16-byte aligned");
  // each 8-channel vector of every token must stay 16-byte aligned
  const int64_t e = dtype == SSD_DTYPE_BF16 ? 2 : 4;
  if (x_stride.batch < 0 || x_stride.token < channels || (x_stride.batch * e) % 16 ||
      (x_stride.token * e) % 16)
    return bad(SSD_ERR_ALIGN,
               "x strides must be multiples of 16 bytes, the token stride >= channels");
  const int64_t nrun = (seqlen + ssd::block::kConvRun - 1) / ssd::block::kConvRun;
  if (nrun > 2147483647LL) return bad(SSD_ERR_UNSUPPORTED, "seqlen too large");
  const ssd::TokStride sx = {x_stride.batch, x_stride.token};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const cudaError_t err =
      dtype == SSD_DTYPE_F32
          ? ssd::block::launch_conv<float>(static_cast<const float*>(x), sx, weight, bias,
                                           seq_idx, batch, seqlen, channels, width, silu,
                                           static_cast<float*>(out), st)
          : ssd::block::launch_conv<__nv_bfloat16>(
                static_cast<const __nv_bfloat16*>(x), sx, weight, bias, seq_idx, batch, seqlen,
                channels, width, silu, static_cast<__nv_bfloat16*>(out), st);
  if (err != cudaSuccess) {
    char m[256];
    snprintf(m, sizeof(m), "causal_conv1d launch: %s", cudaGetErrorString(err));
    return bad(SSD_ERR_CUDA, m);
  }
  return SSD_OK;
}

int ssd_group_rmsnorm(void* y, const float* weight, float eps, int64_t rows, int dim,
                      int group_size, ssd_dtype_t dtype, void* stream) {
  if (dtype != SSD_DTYPE_F32 && dtype != SSD_DTYPE_BF16) return bad(SSD_ERR_ARG, "unknown dtype");
  if (rows < 1 || dim < 1 || group_size < 1 || dim % group_size != 0)
    return bad(SSD_ERR_ARG, "rows, dim >= 1 and group_size dividing dim are required");
  if (group_size % ssd::block::kVec != 0)
    return bad(SSD_ERR_UNSUPPORTED, "group_size must be a multiple of 8");
  if (!(eps >= 0.f)) return bad(SSD_ERR_ARG, "eps must be >= 0");
  if (!y || !weight) return bad(SSD_ERR_NULL, "y and weight are required");
  if (!al16(y)) return bad(SSD_ERR_ALIGN, "y must be 16-byte aligned");
  const int64_t warps = rows * (dim / group_size);
  const int64_t blocks = (warps * 32 + 255) / 256;
  if (blocks > 2147483647LL) return bad(SSD_ERR_UNSUPPORTED, "too many rows");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (dtype == SSD_DTYPE_F32)
    ssd::block::group_rmsnorm_kernel<float><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<float*>(y), weight, eps, rows, dim, group_size);
  else
    ssd::block::group_rmsnorm_kernel<__nv_bfloat16><<<(unsigned)blocks, 256, 0, st>>>(
        static_cast<__nv_bfloat16*>(y), weight, eps, rows, dim, group_size);
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) {
    char m[256];
    snprintf(m, sizeof(m), "group_rmsnorm launch: %s", cudaGetErrorString(err));
    return bad(SSD_ERR_CUDA, m);
  }
  return SSD_OK;
}

}  // extern "C"
