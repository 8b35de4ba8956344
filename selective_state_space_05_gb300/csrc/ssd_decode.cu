// Single-token decode step of the SSD recurrence: the state a prefill left
// (final_states of ssd_scan_fwd) advanced by one token per batch row, in
// place, with the token's output.  Initial / final states are what make
// chunked prefill and speculative decoding possible (state-spaces/mamba PR
// #488); one decode step is the recurrence itself at L = 1:
//   dt' = clamp(softplus(dt + dt_bias)),  h <- exp(dt' A) h + dt' x (outer) B
//   y = h C + D x,  out = y * silu(z)
// HBM-bound on the fp32 state (read and written once).  One CTA per
// (batch row, head), four warps: warp w walks the state rows p = w, w + 4,
// ..., four rows per pass with all their loads in flight first; a warp
// reads a whole row per instruction (lane l: dstate columns
// 4l .. 4l+3, and 4l + 128 .. for dstate 256), keeps its columns of B and
// C in registers, and sums h C over the row with shuffles.
#include <math.h>
#include <stdio.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"

namespace ssd {
namespace decode {

// Q4: column quads per lane (1 for dstate <= 128, else 2); the rows per
// pass shrink as the quads grow, to keep the registers in flight constant.
template <typename T, int Q4>
__global__ void __launch_bounds__(128)
    decode_step_kernel(const T* __restrict__ x, const T* __restrict__ dt,
                       const float* __restrict__ dt_bias, int softplus, int do_clamp, float lo,
                       float hi, const float* __restrict__ A, const T* __restrict__ Bm,
                       const T* __restrict__ Cm, const float* __restrict__ D,
                       const T* __restrict__ z, float* __restrict__ state, int H, int P, int N,
                       int G, T* __restrict__ out) {
  const int bh = blockIdx.x;
  const int b = bh / H, h = bh % H;
  const int g = h / (H / G);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float d = to_f(dt[(int64_t)b * H + h]) + (dt_bias ? dt_bias[h] : 0.f);
  if (softplus) d = d <= 20.f ? log1pf(__expf(d)) : d;
  if (do_clamp) d = fminf(fmaxf(d, lo), hi);
  const float decay = __expf(d * A[h]);
  const T* Bg = Bm + ((int64_t)b * G + g) * N;
  const T* Cg = Cm + ((int64_t)b * G + g) * N;
  // this lane's (up to two) column quads of B and C
  float bq[Q4][4], cq[Q4][4];
  const int nq = N / 4;
#pragma unroll
  for (int k = 0; k < Q4; ++k) {
    const int c4 = lane + 32 * k;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      bq[k][i] = c4 < nq ? to_f(Bg[4 * c4 + i]) : 0.f;
      cq[k][i] = c4 < nq ? to_f(Cg[4 * c4 + i]) : 0.f;
    }
  }
  const T* xr = x + (int64_t)bh * P;
  const T* zr = z ? z + (int64_t)bh * P : nullptr;
  T* orow = out + (int64_t)bh * P;
  // kRows rows per pass: their loads are all in flight before any is used
  constexpr int kRows = 8 / Q4;
  for (int p0 = warp; p0 < P; p0 += 4 * kRows) {
    float4 v[kRows][Q4];
    float xp[kRows];
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int p = p0 + 4 * u;
      xp[u] = p < P ? to_f(xr[p]) : 0.f;
#pragma unroll
      for (int k = 0; k < Q4; ++k) {
        const int c4 = lane + 32 * k;
        if (p < P && c4 < nq)
          v[u][k] = *reinterpret_cast<const float4*>(state + ((int64_t)bh * P + p) * N + 4 * c4);
      }
    }
#pragma unroll
    for (int u = 0; u < kRows; ++u) {
      const int p = p0 + 4 * u;
      if (p >= P) break;   // (uniform across the warp)
      const float dx = d * xp[u];
      float acc = 0.f;
#pragma unroll
      for (int k = 0; k < Q4; ++k) {
        const int c4 = lane + 32 * k;
        if (c4 < nq) {
          float4 w = v[u][k];
          w.x = fmaf(decay, w.x, dx * bq[k][0]);
          w.y = fmaf(decay, w.y, dx * bq[k][1]);
          w.z = fmaf(decay, w.z, dx * bq[k][2]);
          w.w = fmaf(decay, w.w, dx * bq[k][3]);
          *reinterpret_cast<float4*>(state + ((int64_t)bh * P + p) * N + 4 * c4) = w;
          acc = fmaf(w.x, cq[k][0], fmaf(w.y, cq[k][1], fmaf(w.z, cq[k][2], fmaf(w.w, cq[k][3], acc))));
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
      if (lane == 0) {
        float y = acc + (D ? D[h] * xp[u] : 0.f);
        if (zr) {
          const float zz = to_f(zr[p]);
          y *= zz / (1.f + __expf(-zz));
        }
        orow[p] = from_f<T>(y);
      }
    }
  }
}

}  // namespace decode
}  // namespace ssd

extern "C" {

int ssd_decode_step(const void* x, const void* dt, const float* dt_bias, int dt_softplus,
                    float dt_limit_lo, float dt_limit_hi, const float* A, const void* B,
                    const void* C, const float* D, const void* z, float* state, int64_t batch,
                    int nheads, int headdim, int dstate, int ngroups, ssd_dtype_t dtype,
                    void* out, void* stream) {
  if (dtype != SSD_DTYPE_F32 && dtype != SSD_DTYPE_BF16)
    return ssd::set_error(SSD_ERR_ARG, "unknown dtype");
  if (batch < 1 || nheads < 1 || ngroups < 1 || nheads % ngroups != 0)
    return ssd::set_error(SSD_ERR_ARG, "batch, nheads >= 1 and ngroups dividing nheads needed");
  if (headdim < 1 || headdim > 4096)
    return ssd::set_error(SSD_ERR_UNSUPPORTED, "headdim must be in [1, 4096]");
  if (dstate < 8 || dstate > 256 || dstate % 8 != 0)
    return ssd::set_error(SSD_ERR_UNSUPPORTED, "dstate must be a multiple of 8 in [8, 256]");
  if ((int64_t)batch * nheads > 2147483647LL)
    return ssd::set_error(SSD_ERR_UNSUPPORTED, "batch * nheads too large");
  if (!(dt_limit_lo <= dt_limit_hi)) return ssd::set_error(SSD_ERR_ARG, "dt_limit lo > hi");
  if (!x || !dt || !A || !B || !C || !state || !out)
    return ssd::set_error(SSD_ERR_NULL, "x, dt, A, B, C, state and out are required");
  if (((uintptr_t)state & 15u) != 0)
    return ssd::set_error(SSD_ERR_ALIGN, "state must be 16-byte aligned");
  const int clamp = !(dt_limit_lo == 0.f && isinf(dt_limit_hi) && dt_limit_hi > 0.f);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const unsigned grid = (unsigned)(batch * nheads);
  using bf = __nv_bfloat16;
#define SSD_DECODE(T, Q4)                                                                    \
  ssd::decode::decode_step_kernel<T, Q4><<<grid, 128, 0, st>>>(                              \
      static_cast<const T*>(x), static_cast<const T*>(dt), dt_bias, dt_softplus, clamp,      \
      dt_limit_lo, dt_limit_hi, A, static_cast<const T*>(B), static_cast<const T*>(C), D,    \
      static_cast<const T*>(z), state, nheads, headdim, dstate, ngroups, static_cast<T*>(out))
  if (dtype == SSD_DTYPE_F32) {
    if (dstate <= 128) SSD_DECODE(float, 1); else SSD_DECODE(float, 2);
  } else {
    if (dstate <= 128) SSD_DECODE(bf, 1); else SSD_DECODE(bf, 2);
  }
#undef SSD_DECODE
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    char m[256];
    snprintf(m, sizeof(m), "decode_step launch: %s", cudaGetErrorString(e));
    return ssd::set_error(SSD_ERR_CUDA, m);
  }
  return SSD_OK;
}

}  // extern "C"
