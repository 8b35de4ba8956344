// Backward of the SSD chunked-scan forward (fp32): the gradients of a loss
// sum(out * dout) with respect to x, raw dt, dt_bias, A, B, C, D, z and the
// initial states.  The fla-org/flash-linear-attention PR #49 page asks to
// check backward correctness as well as the forward's; the initial-state PR
// (state-spaces/mamba #488) left the backward out.
//
// The adjoint of a linear recurrence is a linear recurrence run backwards in
// time, so every heavy part here is one of the forward's own scans (the
// stage kernels of ssd_simt.cu, with the roles of the operands swapped),
// written in terms of the forward's quantities: dt (processed), a = dt A and
// the decay L_ij = exp(a_{j+1} + ... + a_i) between tokens j <= i of one
// document.  With dy = dout * silu(z) and y the forward output before the gate:
//   g_j  = sum_{i>=j} L_ij (C_i . B_j) dy_i            (time-reversed scan of
//          dy with B' = C, C' = B, value coefficient 1 and the decays
//          shifted by one token: the reversed token of t decays by a_{t+1})
//   dx_j = dt_j g_j + D dy_j
//   dB_j = dt_j sum_{h in group} sum_{i>=j} L_ij (x_j . dy_i) C_i
//          (reversed scan with x' = C, B' = dy, C' = x)
//   dC_i = sum_{h in group} [sum_{j<=i} L_ij dt_j (dy_i . x_j) B_j
//          + exp(cs_i) h0^T dy_i]   (forward scan with x' = B, B' = x, C' = dy)
//   da_k = sum over the pairs j < k <= i of their term
//          P_ij = L_ij (C_i . B_j) dt_j (dy_i . x_j)   (each decays through a_k)
//   ddt  = da A + x . g, then through the clamp, softplus and bias;
//   dA = sum da dt,  dD = sum dy . x,  dz = dout y silu'(z),
//   dh0 = exp(a_0) (final state of the dx scan).
//
// da.  With q_m = dy_m . yo_m - dt_m x_m . go_m (yo, go: y without D x and g,
// each without the diagonal pair), sum_{m>=k} q_m telescopes to da_k, but
// over the whole sequence that sum cancels almost entirely under strong
// decay and its rounding grows with the length.  So the telescoping stops at
// the end of k's chunk: the pairs that cross the boundary after chunk c sum
// exactly to <dH_c, H_c>, H_c the forward state after chunk c and dH_c the
// state of the reversed g scan at the same boundary, so
//   da_k = sum_{m in chunk(k), m >= k} q_m + <dH_c, H_c>.
// The backward runs its scans with its own chunk length (128 on the fp32
// tensor-core stages, else at most kBwdChunk; the result does not depend on
// it), and pads the reversed sequence to whole chunks so that the reversed
// chunk boundaries fall on the forward ones.
#include <math.h>
#include <stdio.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"

namespace ssd {
namespace bwd {

constexpr int kBwdChunk = 64;

__device__ __forceinline__ int64_t chunk_index(int64_t b, int h, int64_t t, int H, int nc, int Q) {
  return (((int64_t)b * H + h) * nc + t / Q) * Q + t % Q;   // [B, H, nc, Q]
}

// Over the reversed index space [B, Lp, H, P] (Lp >= L; reversed token k'
// is forward token t = Lp-1-k', padding where t >= L), four elements per
// thread (H P is a multiple of 4): dy = dout silu(z) (dout without z) in
// forward order, and the reversed copies of dy and x (zero on the padding).
__global__ void reversed_prep_kernel(const float* __restrict__ dout, const float* __restrict__ z,
                                     const float* __restrict__ x, int64_t Bz, int64_t L,
                                     int64_t Lp, int HP, float* __restrict__ dy,
                                     float* __restrict__ dyR, float* __restrict__ xR) {
  const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (r >= Bz * Lp * HP) return;
  const int64_t b = r / (Lp * HP), t = Lp - 1 - (r / HP) % Lp, c = r % HP;
  float4* dyr = reinterpret_cast<float4*>(dyR + r);
  float4* xr = reinterpret_cast<float4*>(xR + r);
  if (t >= L) {
    *dyr = make_float4(0.f, 0.f, 0.f, 0.f);
    *xr = make_float4(0.f, 0.f, 0.f, 0.f);
    return;
  }
  const int64_t i = (b * L + t) * HP + c;
  float4 v = *reinterpret_cast<const float4*>(dout + i);
  if (z) {
    const float4 zz = *reinterpret_cast<const float4*>(z + i);
    v.x *= zz.x / (1.f + __expf(-zz.x));
    v.y *= zz.y / (1.f + __expf(-zz.y));
    v.z *= zz.z / (1.f + __expf(-zz.z));
    v.w *= zz.w / (1.f + __expf(-zz.w));
  }
  *reinterpret_cast<float4*>(dy + i) = v;
  *dyr = v;
  *xr = *reinterpret_cast<const float4*>(x + i);
}

// out[b, k, :] = in[b, Lp-1-k, :] for a [B, L, W] input (zero where
// Lp-1-k >= L): the time-reversed, padded copy.
__global__ void reverse_kernel(const float* __restrict__ in, int64_t Bz, int64_t L, int64_t Lp,
                               int64_t W, float* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= Bz * Lp * W) return;
  const int64_t b = i / (Lp * W), t = Lp - 1 - (i / W) % Lp, c = i % W;
  out[i] = t < L ? in[(b * L + t) * W + c] : 0.f;
}

// The reversed decays aR[b, k', h] = a_{t+1} for the reversed token k' of
// forward token t = Lp-1-k' (0 where t+1 >= L), and seqR[b, k'] = seq[b,
// min(t, L-1)] (the padding continues the last document).
__global__ void reversed_decay_kernel(const float* __restrict__ dtF, const float* __restrict__ A,
                                      const int32_t* __restrict__ seq, int64_t Bz, int64_t L,
                                      int64_t Lp, int H, int nc, int Q, float* __restrict__ aR,
                                      int32_t* __restrict__ seqR) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= Bz * Lp * H) return;
  const int64_t b = i / (Lp * H), t = Lp - 1 - (i / H) % Lp;
  const int h = (int)(i % H);
  aR[i] = t + 1 < L ? dtF[chunk_index(b, h, t + 1, H, nc, Q)] * A[h] : 0.f;
  if (seq && h == 0) seqR[b * Lp + (Lp - 1 - t)] = seq[b * L + (t < L ? t : L - 1)];
}

__global__ void fill_kernel(float* __restrict__ p, int64_t n, float v) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) p[i] = v;
}

// [B, H, P, N] -> [B, H, N, P]
__global__ void transpose_state_kernel(const float* __restrict__ in, int64_t BH, int P, int N,
                                       float* __restrict__ out) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= BH * P * N) return;
  const int64_t bh = i / ((int64_t)P * N);
  const int p = (int)((i / N) % P), n = (int)(i % N);
  out[(bh * N + n) * P + p] = in[i];
}

// One block per (b, t): C . B once per group (in shared memory), then one
// warp per head in turn (lanes over P): the diagonal added back (g = go +
// (C.B) dy, y = yo + dt x (C.B) + D x), dx, dz, and the per-token sums q,
// x . g and dy . x.  goR is in reversed order over Lp tokens.
__global__ void __launch_bounds__(256) token_grads_kernel(
    const float* __restrict__ goR, const float* __restrict__ yo, const float* __restrict__ x,
    const float* __restrict__ dout, const float* __restrict__ z, const float* __restrict__ Bm,
    const float* __restrict__ Cm, const float* __restrict__ D, const float* __restrict__ dtF,
    int64_t L, int64_t Lp, int H, int P, int N, int G, int nc, int Q, float* __restrict__ dx,
    float* __restrict__ dz, float* __restrict__ q, float* __restrict__ xg,
    float* __restrict__ dyx) {
  extern __shared__ float cb_s[];   // [G]
  const int64_t b = blockIdx.x / L, t = blockIdx.x % L;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int g = warp; g < G; g += 8) {
    const int64_t bg = ((b * L + t) * G + g) * N;
    float cb = 0.f;
    for (int n = lane; n < N; n += 32) cb = fmaf(Cm[bg + n], Bm[bg + n], cb);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) cb += __shfl_xor_sync(0xffffffffu, cb, off);
    if (lane == 0) cb_s[g] = cb;
  }
  __syncthreads();
  for (int h = warp; h < H; h += 8) {
    const float cb = cb_s[h / (H / G)];
    const float dt = dtF[chunk_index(b, h, t, H, nc, Q)];
    const float Dh = D ? D[h] : 0.f;
    const int64_t w = (b * L + t) * H + h;
    const int64_t base = w * P, rbase = ((b * Lp + (Lp - 1 - t)) * H + h) * P;
    float s_q = 0.f, s_xg = 0.f, s_dyx = 0.f;
    for (int p = 2 * lane; p < P; p += 64) {   // two consecutive elements per lane
      const float2 xv = *reinterpret_cast<const float2*>(x + base + p);
      const float2 go = *reinterpret_cast<const float2*>(goR + rbase + p);
      const float2 yv = *reinterpret_cast<const float2*>(yo + base + p);
      float2 dyv = *reinterpret_cast<const float2*>(dout + base + p);
      if (z) {
        const float2 zz = *reinterpret_cast<const float2*>(z + base + p);
        const float s0 = 1.f / (1.f + __expf(-zz.x)), s1 = 1.f / (1.f + __expf(-zz.y));
        const float y0 = yv.x + (dt * cb + Dh) * xv.x, y1 = yv.y + (dt * cb + Dh) * xv.y;
        *reinterpret_cast<float2*>(dz + base + p) =
            make_float2(dyv.x * y0 * s0 * (1.f + zz.x * (1.f - s0)),
                        dyv.y * y1 * s1 * (1.f + zz.y * (1.f - s1)));
        dyv.x *= zz.x * s0;
        dyv.y *= zz.y * s1;
      }
      const float g0 = fmaf(cb, dyv.x, go.x), g1 = fmaf(cb, dyv.y, go.y);
      *reinterpret_cast<float2*>(dx + base + p) =
          make_float2(fmaf(dt, g0, Dh * dyv.x), fmaf(dt, g1, Dh * dyv.y));
      s_q += dyv.x * yv.x - dt * xv.x * go.x + dyv.y * yv.y - dt * xv.y * go.y;
      s_xg = fmaf(xv.x, g0, fmaf(xv.y, g1, s_xg));
      s_dyx = fmaf(dyv.x, xv.x, fmaf(dyv.y, xv.y, s_dyx));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      s_q += __shfl_xor_sync(0xffffffffu, s_q, off);
      s_xg += __shfl_xor_sync(0xffffffffu, s_xg, off);
      s_dyx += __shfl_xor_sync(0xffffffffu, s_dyx, off);
    }
    if (lane == 0) {
      q[w] = s_q;
      xg[w] = s_xg;
      dyx[w] = s_dyx;
    }
  }
}

// dB[b,t,g,n] = sum_{h in g} dt[b,t,h] oB[b, Lp-1-t, h, n] (oB reversed);
// dC[b,t,g,n] = sum_{h in g} oC[b, t, h, n].
__global__ void group_grads_kernel(const float* __restrict__ oB, const float* __restrict__ oC,
                                   const float* __restrict__ dtF, int64_t Bz, int64_t L,
                                   int64_t Lp, int H, int G, int N, int nc, int Q,
                                   float* __restrict__ dB, float* __restrict__ dC) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= Bz * L * G * N) return;
  const int64_t b = i / (L * G * N), t = (i / ((int64_t)G * N)) % L;
  const int g = (int)((i / N) % G), n = (int)(i % N);
  const int rep = H / G;
  float sb = 0.f, sc = 0.f;
  for (int h = g * rep; h < (g + 1) * rep; ++h) {
    sb += dtF[chunk_index(b, h, t, H, nc, Q)] * oB[((b * Lp + (Lp - 1 - t)) * H + h) * N + n];
    sc += oC[((b * L + t) * H + h) * N + n];
  }
  dB[i] = sb;
  dC[i] = sc;
}

// The boundary term after chunk c, one block per (c, h, b):
// bnd[b, h, c] = <dH_c, H_c> with H_c = the forward prev state of chunk c+1
// and dH_c = exp(a at the first token of chunk c+1) times the reversed prev
// state of reversed chunk nc-1-c (zero across a document start and after
// the last chunk).
__global__ void __launch_bounds__(256) boundary_kernel(
    const float* __restrict__ prevF, const float* __restrict__ prevR,
    const int32_t* __restrict__ segF, const float* __restrict__ dtF, const float* __restrict__ A,
    int H, int PN, int nc, int Q, float* __restrict__ bnd) {
  __shared__ float part[8];
  const int c = blockIdx.x, h = blockIdx.y;
  const int64_t b = blockIdx.z;
  float* out = bnd + ((int64_t)b * H + h) * nc + c;
  if (c == nc - 1 || (segF && segF[((int64_t)b * nc + c + 1) * Q] != 0)) {
    if (threadIdx.x == 0) *out = 0.f;
    return;
  }
  const float4* hf =
      reinterpret_cast<const float4*>(prevF + (((int64_t)b * nc + c + 1) * H + h) * (int64_t)PN);
  const float4* hr = reinterpret_cast<const float4*>(
      prevR + (((int64_t)b * nc + (nc - 1 - c)) * H + h) * (int64_t)PN);
  float s = 0.f;
  for (int e = threadIdx.x; e < PN / 4; e += 256) {
    const float4 u = hf[e], v = hr[e];
    s = fmaf(u.x, v.x, fmaf(u.y, v.y, fmaf(u.z, v.z, fmaf(u.w, v.w, s))));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if ((threadIdx.x & 31) == 0) part[threadIdx.x >> 5] = s;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < 8; ++w) t += part[w];
    *out = __expf(dtF[chunk_index(b, h, (int64_t)(c + 1) * Q, H, nc, Q)] * A[h]) * t;
  }
}

// One warp per (b, h, chunk): da = the boundary term after the chunk plus the
// suffix sum of q inside the chunk, then ddt = da A + x . g through clamp,
// softplus and bias; dA, d dt_bias and dD summed (atomics across warps).
__global__ void dt_grads_kernel(const float* __restrict__ q, const float* __restrict__ xg,
                                const float* __restrict__ dyx, const float* __restrict__ bnd,
                                const float* __restrict__ dt_raw,
                                const float* __restrict__ dt_bias, int softplus, int do_clamp,
                                float lo, float hi, const float* __restrict__ A,
                                const float* __restrict__ dtF, int64_t Bz, int64_t L, int H,
                                int nc, int Q, float* __restrict__ ddt, float* __restrict__ dA,
                                float* __restrict__ dbias, float* __restrict__ dD) {
  const int64_t w = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (w >= Bz * H * nc) return;
  const int c = (int)(w % nc);
  const int h = (int)((w / nc) % H);
  const int64_t b = w / ((int64_t)nc * H);
  const float Ah = A[h], bias = dt_bias ? dt_bias[h] : 0.f;
  const int64_t start = (int64_t)c * Q;
  const int64_t n = (L - start) < Q ? (L - start) : Q;
  float carry = bnd[w], sA = 0.f, sbias = 0.f, sD = 0.f;
  for (int64_t t0 = start + ((n - 1) / 32) * 32; t0 >= start; t0 -= 32) {   // last 32 first
    const int64_t t = t0 + lane;
    const bool ok = t < start + n;
    const int64_t idx = (b * L + t) * H + h;
    const float qv = ok ? q[idx] : 0.f;
    float s = qv;   // suffix sum over the lanes >= this one
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float o = __shfl_down_sync(0xffffffffu, s, off);
      if (lane + off < 32) s += o;
    }
    const float da = s + carry;
    carry += __shfl_sync(0xffffffffu, s, 0);
    if (ok) {
      const float dt = dtF[chunk_index(b, h, t, H, nc, Q)];
      sA = fmaf(da, dt, sA);
      // back through clamp (passes where lo <= v <= hi), softplus and bias
      const float raw = dt_raw[idx] + bias;
      float g = fmaf(da, Ah, xg[idx]);
      if (do_clamp) {
        const float v = softplus ? (raw <= 20.f ? log1pf(__expf(raw)) : raw) : raw;
        g = (v >= lo && v <= hi) ? g : 0.f;
      }
      if (softplus) g *= 1.f / (1.f + __expf(-raw));
      ddt[idx] = g;
      sbias += g;
      sD += dyx[idx];
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    sA += __shfl_xor_sync(0xffffffffu, sA, off);
    sbias += __shfl_xor_sync(0xffffffffu, sbias, off);
    sD += __shfl_xor_sync(0xffffffffu, sD, off);
  }
  if (lane == 0) {
    atomicAdd(dA + h, sA);
    if (dbias) atomicAdd(dbias + h, sbias);
    if (dD) atomicAdd(dD + h, sD);
  }
}

// dh0 = exp(a_0) F, F the final state of the reversed dx scan ([B,H,P,N]).
__global__ void dh0_kernel(const float* __restrict__ F, const float* __restrict__ dtF,
                           const float* __restrict__ A, int64_t Bz, int H, int PN, int nc, int Q,
                           float* __restrict__ dh0) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= Bz * H * PN) return;
  const int64_t bh = i / PN;
  const int h = (int)(bh % H);
  dh0[i] = __expf(dtF[chunk_index(bh / H, h, 0, H, nc, Q)] * A[h]) * F[i];
}

// bf16 <-> fp32 copies for the bf16 entry point: four elements per thread,
// the last partial group one by one.
__global__ void bf16_to_f32_kernel(const __nv_bfloat16* __restrict__ in, int64_t n,
                                   float* __restrict__ out) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i >= n) return;
  if (i + 4 <= n) {
    const __nv_bfloat162 a = reinterpret_cast<const __nv_bfloat162*>(in + i)[0];
    const __nv_bfloat162 b = reinterpret_cast<const __nv_bfloat162*>(in + i)[1];
    const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
    *reinterpret_cast<float4*>(out + i) = make_float4(fa.x, fa.y, fb.x, fb.y);
  } else {
    for (int64_t k = i; k < n; ++k) out[k] = __bfloat162float(in[k]);
  }
}
__global__ void f32_to_bf16_kernel(const float* __restrict__ in, int64_t n,
                                   __nv_bfloat16* __restrict__ out) {
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i >= n) return;
  if (i + 4 <= n) {
    const float4 v = *reinterpret_cast<const float4*>(in + i);
    reinterpret_cast<__nv_bfloat162*>(out + i)[0] = __floats2bfloat162_rn(v.x, v.y);
    reinterpret_cast<__nv_bfloat162*>(out + i)[1] = __floats2bfloat162_rn(v.z, v.w);
  } else {
    for (int64_t k = i; k < n; ++k) out[k] = __float2bfloat16_rn(in[k]);
  }
}

// The backward's own chunk length: 128 where its scans (headdim x dstate
// and the swapped dstate x headdim) take the fp32 tensor-core stages,
// otherwise at most kBwdChunk (shorter in-chunk sums, see above).
int bwd_chunk(int chunk_size, int P, int N) {
  const bool tc = (P == 64 || P == 128) && (N == 64 || N == 128) && (P == 128 || N == 128);
  if (tc && chunk_size >= 128) return 128;
  return chunk_size < kBwdChunk ? chunk_size : kBwdChunk;
}

// Workspace pieces, 256-byte aligned.  Reversed arrays span Lp = nc Qb tokens.
struct BwdLayout {
  size_t dtF, csF, segF, statesF, yo, dy, dyR, xR, CR, BR, aR, seqR, csR, dtRo, segR, ones,
      states1, finR, goR, states2, oB, h0T, oC, q, xg, dyx, bnd, cb, cbT, tgB, tgCR, total;
};

BwdLayout bwd_layout(int64_t Bz, int64_t L, int H, int P, int N, int G, int Q) {
  const int64_t nc = (L + Q - 1) / Q, Lp = nc * Q;
  const size_t chunk = (size_t)Bz * H * nc * Q, seg = (size_t)Bz * nc * Q;
  const size_t xs = (size_t)Bz * L * H * P, xsR = (size_t)Bz * Lp * H * P;
  const size_t bsR = (size_t)Bz * Lp * G * N, hs = (size_t)Bz * L * H * N;
  const size_t hsR = (size_t)Bz * Lp * H * N, st = (size_t)Bz * nc * H * P * N;
  const size_t tok = (size_t)Bz * L * H;
  BwdLayout l;
  size_t o = 0;
  auto take = [&](size_t elems) {   // 4-byte elements
    const size_t at = o;
    o = (o + elems * 4 + 255) / 256 * 256;
    return at;
  };
  l.dtF = take(chunk);
  l.csF = take(chunk);
  l.segF = take(seg);
  l.statesF = take(st);
  l.yo = take(xs);
  l.dy = take(xs);
  l.dyR = take(xsR);
  l.xR = take(xsR);
  l.CR = take(bsR);
  l.BR = take(bsR);
  l.aR = take((size_t)Bz * Lp * H);
  l.seqR = take((size_t)Bz * Lp);
  l.csR = take(chunk);
  l.dtRo = take(chunk);
  l.segR = take(seg);
  l.ones = take(chunk);
  l.states1 = take(st);
  l.finR = take((size_t)Bz * H * P * N);
  l.goR = take(xsR);
  l.states2 = take(st);
  l.oB = take(hsR);
  l.h0T = take((size_t)Bz * H * P * N);
  l.oC = take(hs);
  l.q = take(tok);
  l.xg = take(tok);
  l.dyx = take(tok);
  l.bnd = take((size_t)Bz * H * nc);
  // C B^T per (batch, chunk, group) and its transpose, shared by the heads
  // (used where the scans take the fp32 tensor-core stages, 128-token chunks)
  const size_t cbn = Q == 128 ? (size_t)Bz * nc * G * Q * Q : 0;
  l.cb = take(cbn);
  l.cbT = take(cbn);
  // B and the reversed C as chunk_state's pre-split A tiles (dstate 128)
  const size_t tgn = (Q == 128 && N == 128) ? (size_t)Bz * nc * G * 8 * 4096 : 0;
  l.tgB = take(tgn);
  l.tgCR = take(tgn);
  l.total = o;
  return l;
}

unsigned blocks_for(int64_t n, int per) { return (unsigned)((n + per - 1) / per); }

}  // namespace bwd
}  // namespace ssd

namespace {

int bfail(int code, const char* msg) { return ssd::set_error(code, msg); }

bool bwd_sizes_ok(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
                  int chunk) {
  auto pow2 = [](int v, int lo, int hi) {
    for (int s = lo; s <= hi; s *= 2)
      if (v == s) return true;
    return false;
  };
  return batch >= 1 && batch <= 65535 && seqlen >= 1 && nheads >= 1 && nheads <= 65535 &&
         ngroups >= 1 && ngroups <= 8192 && nheads % ngroups == 0 && pow2(headdim, 16, 128) &&
         pow2(dstate, 16, 128) &&
         pow2(chunk, 16, 256) && (seqlen + chunk - 1) / chunk * batch <= 2147483647LL;
}

ssd::Dims dims_of(int64_t Bz, int64_t L, int H, int P, int N, int G, int Q) {
  ssd::Dims d;
  d.batch = Bz;
  d.seqlen = L;
  d.nheads = H;
  d.headdim = P;
  d.dstate = N;
  d.ngroups = G;
  d.chunk = Q;
  d.nchunks = (int)((L + Q - 1) / Q);
  d.sx = {L * H * P, (int64_t)H * P};
  d.sz = d.sx;
  d.sdt = {L * H, H};
  d.sB = {L * G * N, (int64_t)G * N};
  d.sC = d.sB;
  return d;
}

}  // namespace

extern "C" {

size_t ssd_scan_bwd_workspace_bytes(int64_t batch, int64_t seqlen, int nheads, int headdim,
                                    int dstate, int ngroups, int chunk_size) {
  if (!bwd_sizes_ok(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size)) return 0;
  return ssd::bwd::bwd_layout(batch, seqlen, nheads, headdim, dstate, ngroups,
                              ssd::bwd::bwd_chunk(chunk_size, headdim, dstate))
      .total;
}

int ssd_scan_bwd(const float* x, const float* dt, const float* dt_bias, int dt_softplus,
                 float dt_limit_lo, float dt_limit_hi, const float* A, const float* B,
                 const float* C, const float* D, const float* z, const float* initial_states,
                 const int32_t* seq_idx, const float* dout, int64_t batch, int64_t seqlen,
                 int nheads, int headdim, int dstate, int ngroups, int chunk_size, float* dx,
                 float* ddt, float* d_dt_bias, float* dA, float* dB, float* dC, float* dD,
                 float* dz, float* d_initial_states, void* workspace, size_t workspace_bytes,
                 void* stream) {
  using namespace ssd::bwd;
  if (!bwd_sizes_ok(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size))
    return bfail(SSD_ERR_UNSUPPORTED,
                 "ssd_scan_bwd: headdim and dstate in {16, 32, 64, 128}, chunk_size a power of "
                 "two in [16, 256], ngroups dividing nheads and at most 8192");
  if (!(dt_limit_lo <= dt_limit_hi)) return bfail(SSD_ERR_ARG, "dt_limit lo > hi");
  if (!x || !dt || !A || !B || !C || !dout || !dx || !ddt || !dA || !dB || !dC || !workspace)
    return bfail(SSD_ERR_NULL, "x, dt, A, B, C, dout, dx, ddt, dA, dB, dC, workspace required");
  if (z && !dz) return bfail(SSD_ERR_NULL, "dz is required with z");
  const void* ptrs[] = {x, dt, dt_bias, A, B, C, D, z, initial_states, seq_idx, dout, dx, ddt,
                        d_dt_bias, dA, dB, dC, dD, dz, d_initial_states, workspace};
  for (const void* p : ptrs)
    if (((uintptr_t)p & 15u) != 0) return bfail(SSD_ERR_ALIGN, "pointers must be 16-byte aligned");
  const int64_t Bz = batch, L = seqlen;
  const int H = nheads, P = headdim, N = dstate, G = ngroups, Q = bwd_chunk(chunk_size, P, N);
  const BwdLayout lay = bwd_layout(Bz, L, H, P, N, G, Q);
  if (workspace_bytes < lay.total) {
    char m[160];
    snprintf(m, sizeof(m), "workspace of %zu bytes < %zu needed", workspace_bytes, lay.total);
    return bfail(SSD_ERR_WORKSPACE, m);
  }
  char* ws = static_cast<char*>(workspace);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  auto I = [&](size_t off) { return reinterpret_cast<int32_t*>(ws + off); };
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const ssd::Dims d = dims_of(Bz, L, H, P, N, G, Q);
  const int nc = d.nchunks;
  const int64_t Lp = (int64_t)nc * Q;
  const ssd::Dims dR = dims_of(Bz, Lp, H, P, N, G, Q);   // reversed, padded to whole chunks
  // the swapped scans: headdim' = dstate, dstate' = headdim, one group per
  // head; their x' is the per-group B (or reversed C), read by every head of
  // the group (xrep)
  ssd::Dims ds = dims_of(Bz, L, H, N, P, H, Q);
  ds.sx = {L * G * N, (int64_t)G * N};
  ds.xrep = H / G;
  ssd::Dims dsR = dims_of(Bz, Lp, H, N, P, H, Q);
  dsR.sx = {Lp * G * N, (int64_t)G * N};
  dsR.xrep = H / G;
  const int clamp = !(dt_limit_lo == 0.f && isinf(dt_limit_hi) && dt_limit_hi > 0.f);
  const bool seq = seq_idx != nullptr;
  int32_t* segF = seq ? I(lay.segF) : nullptr;
  int32_t* segR = seq ? I(lay.segR) : nullptr;
  cudaError_t e = cudaSuccess;
  auto ok = [&]() { return e == cudaSuccess && (e = cudaGetLastError()) == cudaSuccess; };

  // forward quantities: stage 1, the chunk states H, and y before the gate
  // without D x and without the diagonal (strict)
  e = ssd::launch_dt_cumsum<float>(dt, dt_bias, dt_softplus, dt_limit_lo, dt_limit_hi, clamp, A,
                                   seq_idx, d, F(lay.dtF), F(lay.csF), segF, st);
  // chunk_state on tensor cores with the per-group operand pre-split once:
  // B for the forward-orientation scans and (headdim 64) the dC scan, the
  // reversed C for the g scan and (headdim 64) the dB scan
  const bool tiles = Q == 128 && N == 128 && ssd::chunk_state_tc32_fits(x, B, d);
  const bool tiles_swapped = tiles && P == 64;
  if (e == cudaSuccess && tiles)
    e = ssd::launch_group_tiles_tc32(B, d.sB, G, Bz, L, nc, F(lay.tgB), st);
  auto state = [&](const float* xo, const float* Bo, const float* dto, const float* cso,
                   const int32_t* sgo, const ssd::Dims& dd, float* out, const float* tg) {
    return tg ? ssd::launch_chunk_state_tc32(xo, Bo, dto, cso, sgo, dd, out, st, tg)
              : ssd::launch_chunk_state<float>(xo, Bo, dto, cso, sgo, dd, out, st);
  };
  if (e == cudaSuccess)
    e = state(x, B, F(lay.dtF), F(lay.csF), segF, d, F(lay.statesF),
              tiles ? F(lay.tgB) : nullptr);
  if (e == cudaSuccess)
    e = ssd::launch_state_passing(F(lay.statesF), F(lay.csF), segF, initial_states, nullptr, d,
                                  st);
  // C B^T once per (batch, chunk, group) for the two scans in the forward
  // orientation (the g scan reads its transpose, reversed)
  const bool shared_cb = Q == 128 && ssd::cb_tc32_fits(B, C, d) &&
                         ssd::chunk_scan_tc32_fits(x, B, C, nullptr, d);
  if (e == cudaSuccess && shared_cb)
    e = ssd::launch_cb_tc32(B, C, d, F(lay.cb), F(lay.cbT), st);
  if (e == cudaSuccess)
    e = shared_cb ? ssd::launch_chunk_scan_tc32(x, B, C, F(lay.dtF), F(lay.csF), segF,
                                                F(lay.statesF), nullptr, nullptr, d, F(lay.yo),
                                                st, 1, F(lay.cb), 0)
                  : ssd::launch_chunk_scan<float>(x, B, C, F(lay.dtF), F(lay.csF), segF,
                                                  F(lay.statesF), nullptr, nullptr, d, F(lay.yo),
                                                  st, 1);
  // gate, reversed copies, the reversed decays
  if (e == cudaSuccess) {
    reversed_prep_kernel<<<blocks_for(Bz * Lp * H * P / 4, 256), 256, 0, st>>>(
        dout, z, x, Bz, L, Lp, H * P, F(lay.dy), F(lay.dyR), F(lay.xR));
    reverse_kernel<<<blocks_for(Bz * Lp * G * N, 256), 256, 0, st>>>(C, Bz, L, Lp,
                                                                     (int64_t)G * N, F(lay.CR));
    reverse_kernel<<<blocks_for(Bz * Lp * G * N, 256), 256, 0, st>>>(B, Bz, L, Lp,
                                                                     (int64_t)G * N, F(lay.BR));
    reversed_decay_kernel<<<blocks_for(Bz * Lp * H, 256), 256, 0, st>>>(
        F(lay.dtF), A, seq_idx, Bz, L, Lp, H, nc, Q, F(lay.aR), seq ? I(lay.seqR) : nullptr);
    fill_kernel<<<blocks_for((int64_t)H, 256), 256, 0, st>>>(F(lay.q), H, 1.f);   // A' = 1
    fill_kernel<<<blocks_for(Bz * H * (int64_t)nc * Q, 256), 256, 0, st>>>(
        F(lay.ones), Bz * H * (int64_t)nc * Q, 1.f);
    ok();
  }
  if (e == cudaSuccess && tiles)
    e = ssd::launch_group_tiles_tc32(F(lay.CR), dR.sC, G, Bz, Lp, nc, F(lay.tgCR), st);
  // stage 1 of the reversed scans: cumsum of the shifted decays (A' = 1, no softplus)
  if (e == cudaSuccess)
    e = ssd::launch_dt_cumsum<float>(F(lay.aR), nullptr, 0, 0.f, INFINITY, 0, F(lay.q),
                                     seq ? I(lay.seqR) : nullptr, dR, F(lay.dtRo), F(lay.csR),
                                     segR, st);
  // g without the diagonal: reversed strict scan of dy with B' = C, C' = B,
  // value coefficient 1; its chunk states are the dH of the boundaries
  if (e == cudaSuccess)
    e = state(F(lay.dyR), F(lay.CR), F(lay.ones), F(lay.csR), segR, dR, F(lay.states1),
              tiles ? F(lay.tgCR) : nullptr);
  if (e == cudaSuccess)
    e = ssd::launch_state_passing(F(lay.states1), F(lay.csR), segR, nullptr, F(lay.finR), dR,
                                  st);
  if (e == cudaSuccess)
    e = shared_cb && ssd::chunk_scan_tc32_fits(F(lay.dyR), F(lay.CR), F(lay.BR), nullptr, dR)
            ? ssd::launch_chunk_scan_tc32(F(lay.dyR), F(lay.CR), F(lay.BR), F(lay.ones),
                                          F(lay.csR), segR, F(lay.states1), nullptr, nullptr, dR,
                                          F(lay.goR), st, 1, F(lay.cbT), 1)
            : ssd::launch_chunk_scan<float>(F(lay.dyR), F(lay.CR), F(lay.BR), F(lay.ones),
                                            F(lay.csR), segR, F(lay.states1), nullptr, nullptr,
                                            dR, F(lay.goR), st, 1);
  if (e == cudaSuccess) {
    boundary_kernel<<<dim3((unsigned)nc, (unsigned)H, (unsigned)Bz), 256, 0, st>>>(
        F(lay.statesF), F(lay.states1), segF, F(lay.dtF), A, H, P * N, nc, Q, F(lay.bnd));
    ok();
  }
  // dB before the dt factor: reversed scan with x' = C (per group), B' = dy,
  // C' = x
  if (e == cudaSuccess)
    e = state(F(lay.CR), F(lay.dyR), F(lay.ones), F(lay.csR), segR, dsR, F(lay.states2),
              tiles_swapped ? F(lay.tgCR) : nullptr);
  if (e == cudaSuccess)
    e = ssd::launch_state_passing(F(lay.states2), F(lay.csR), segR, nullptr, nullptr, dsR, st);
  if (e == cudaSuccess)
    e = ssd::launch_chunk_scan<float>(F(lay.CR), F(lay.dyR), F(lay.xR), F(lay.ones), F(lay.csR),
                                      segR, F(lay.states2), nullptr, nullptr, dsR, F(lay.oB), st);
  // dC per head: forward scan with x' = B (per group), B' = x, C' = dy,
  // initial state h0^T
  if (e == cudaSuccess && initial_states) {
    transpose_state_kernel<<<blocks_for(Bz * H * (int64_t)P * N, 256), 256, 0, st>>>(
        initial_states, Bz * H, P, N, F(lay.h0T));
    ok();
  }
  if (e == cudaSuccess)
    e = state(B, x, F(lay.dtF), F(lay.csF), segF, ds, F(lay.states2),
              tiles_swapped ? F(lay.tgB) : nullptr);
  if (e == cudaSuccess)
    e = ssd::launch_state_passing(F(lay.states2), F(lay.csF), segF,
                                  initial_states ? F(lay.h0T) : nullptr, nullptr, ds, st);
  if (e == cudaSuccess)
    e = ssd::launch_chunk_scan<float>(B, x, F(lay.dy), F(lay.dtF), F(lay.csF), segF,
                                      F(lay.states2), nullptr, nullptr, ds, F(lay.oC), st);
  // the per-token, per-group and per-head gradients
  if (e == cudaSuccess) {
    token_grads_kernel<<<(unsigned)(Bz * L), 256, G * sizeof(float), st>>>(
        F(lay.goR), F(lay.yo), x, dout, z, B, C, D, F(lay.dtF), L, Lp, H, P, N, G, nc, Q, dx, dz,
        F(lay.q), F(lay.xg), F(lay.dyx));
    group_grads_kernel<<<blocks_for(Bz * L * G * N, 256), 256, 0, st>>>(
        F(lay.oB), F(lay.oC), F(lay.dtF), Bz, L, Lp, H, G, N, nc, Q, dB, dC);
    e = cudaMemsetAsync(dA, 0, H * sizeof(float), st);
    if (e == cudaSuccess && d_dt_bias) e = cudaMemsetAsync(d_dt_bias, 0, H * sizeof(float), st);
    if (e == cudaSuccess && dD) e = cudaMemsetAsync(dD, 0, H * sizeof(float), st);
  }
  if (e == cudaSuccess) {
    dt_grads_kernel<<<blocks_for(Bz * H * (int64_t)nc * 32, 256), 256, 0, st>>>(
        F(lay.q), F(lay.xg), F(lay.dyx), F(lay.bnd), dt, dt_bias, dt_softplus, clamp,
        dt_limit_lo, dt_limit_hi, A, F(lay.dtF), Bz, L, H, nc, Q, ddt, dA, d_dt_bias, dD);
    if (d_initial_states)
      dh0_kernel<<<blocks_for(Bz * H * (int64_t)P * N, 256), 256, 0, st>>>(
          F(lay.finR), F(lay.dtF), A, Bz, H, P * N, nc, Q, d_initial_states);
    ok();
  }
  if (e != cudaSuccess) {
    char m[200];
    snprintf(m, sizeof(m), "ssd_scan_bwd launch: %s", cudaGetErrorString(e));
    return bfail(SSD_ERR_CUDA, m);
  }
  return SSD_OK;
}


// The bf16 entry point's extra workspace (after the fp32 backward's): fp32
// copies of x, dt, B, C, z, dout and the fp32 gradients before their bf16
// copies.
namespace {
struct ExLayout {
  size_t x, dt, B, C, z, dout, dx, ddt, dB, dC, dz, total;
};
ExLayout ex_layout(size_t base, int64_t Bz, int64_t L, int H, int P, int N, int G) {
  const size_t xs = (size_t)Bz * L * H * P, ts = (size_t)Bz * L * H, bs = (size_t)Bz * L * G * N;
  ExLayout e;
  size_t o = (base + 255) / 256 * 256;
  auto take = [&](size_t elems) {
    const size_t at = o;
    o = (o + elems * 4 + 255) / 256 * 256;
    return at;
  };
  e.x = take(xs);
  e.dt = take(ts);
  e.B = take(bs);
  e.C = take(bs);
  e.z = take(xs);
  e.dout = take(xs);
  e.dx = take(xs);
  e.ddt = take(ts);
  e.dB = take(bs);
  e.dC = take(bs);
  e.dz = take(xs);
  e.total = o;
  return e;
}
}  // namespace

size_t ssd_scan_bwd_ex_workspace_bytes(int64_t batch, int64_t seqlen, int nheads, int headdim,
                                       int dstate, int ngroups, int chunk_size,
                                       ssd_dtype_t dtype) {
  const size_t base = ssd_scan_bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate,
                                                   ngroups, chunk_size);
  if (base == 0) return 0;
  if (dtype == SSD_DTYPE_F32) return base;
  if (dtype != SSD_DTYPE_BF16) return 0;
  return ex_layout(base, batch, seqlen, nheads, headdim, dstate, ngroups).total;
}

int ssd_scan_bwd_ex(const void* x, const void* dt, const float* dt_bias, int dt_softplus,
                    float dt_limit_lo, float dt_limit_hi, const float* A, const void* B,
                    const void* C, const float* D, const void* z, const float* initial_states,
                    const int32_t* seq_idx, const void* dout, int64_t batch, int64_t seqlen,
                    int nheads, int headdim, int dstate, int ngroups, int chunk_size,
                    ssd_dtype_t dtype, void* dx, void* ddt, float* d_dt_bias, float* dA,
                    void* dB, void* dC, float* dD, void* dz, float* d_initial_states,
                    void* workspace, size_t workspace_bytes, void* stream) {
  using namespace ssd::bwd;
  using bf = __nv_bfloat16;
  if (dtype == SSD_DTYPE_F32)
    return ssd_scan_bwd(static_cast<const float*>(x), static_cast<const float*>(dt), dt_bias,
                        dt_softplus, dt_limit_lo, dt_limit_hi, A, static_cast<const float*>(B),
                        static_cast<const float*>(C), D, static_cast<const float*>(z),
                        initial_states, seq_idx, static_cast<const float*>(dout), batch, seqlen,
                        nheads, headdim, dstate, ngroups, chunk_size, static_cast<float*>(dx),
                        static_cast<float*>(ddt), d_dt_bias, dA, static_cast<float*>(dB),
                        static_cast<float*>(dC), dD, static_cast<float*>(dz), d_initial_states,
                        workspace, workspace_bytes, stream);
  if (dtype != SSD_DTYPE_BF16) return bfail(SSD_ERR_ARG, "unknown dtype");
  const size_t base = ssd_scan_bwd_workspace_bytes(batch, seqlen, nheads, headdim, dstate,
                                                   ngroups, chunk_size);
  if (base == 0)
    return bfail(SSD_ERR_UNSUPPORTED,
                 "ssd_scan_bwd_ex: headdim and dstate in {16, 32, 64, 128}, chunk_size a power "
                 "of two in [16, 256], ngroups dividing nheads and at most 8192");
  if (!x || !dt || !A || !B || !C || !dout || !dx || !ddt || !dA || !dB || !dC || !workspace)
    return bfail(SSD_ERR_NULL, "x, dt, A, B, C, dout, dx, ddt, dA, dB, dC, workspace required");
  if (z && !dz) return bfail(SSD_ERR_NULL, "dz is required with z");
  const void* ptrs[] = {x, dt, B, C, z, dout, dx, ddt, dB, dC, dz, workspace};
  for (const void* p : ptrs)
    if (((uintptr_t)p & 15u) != 0) return bfail(SSD_ERR_ALIGN, "pointers must be 16-byte aligned");
  const ExLayout ex = ex_layout(base, batch, seqlen, nheads, headdim, dstate, ngroups);
  if (workspace_bytes < ex.total) {
    char m[160];
    snprintf(m, sizeof(m), "workspace of %zu bytes < %zu needed", workspace_bytes, ex.total);
    return bfail(SSD_ERR_WORKSPACE, m);
  }
  char* ws = static_cast<char*>(workspace);
  auto F = [&](size_t off) { return reinterpret_cast<float*>(ws + off); };
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t xs = batch * seqlen * nheads * headdim, ts = batch * seqlen * nheads;
  const int64_t bs = batch * seqlen * ngroups * dstate;
  auto up = [&](const void* in, int64_t n, size_t off) {
    bf16_to_f32_kernel<<<blocks_for((n + 3) / 4, 256), 256, 0, st>>>(static_cast<const bf*>(in),
                                                                    n, F(off));
  };
  auto down = [&](size_t off, int64_t n, void* out) {
    f32_to_bf16_kernel<<<blocks_for((n + 3) / 4, 256), 256, 0, st>>>(F(off), n,
                                                                    static_cast<bf*>(out));
  };
  up(x, xs, ex.x);
  up(dt, ts, ex.dt);
  up(B, bs, ex.B);
  up(C, bs, ex.C);
  if (z) up(z, xs, ex.z);
  up(dout, xs, ex.dout);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    char m[200];
    snprintf(m, sizeof(m), "ssd_scan_bwd_ex launch: %s", cudaGetErrorString(e));
    return bfail(SSD_ERR_CUDA, m);
  }
  const int rc = ssd_scan_bwd(F(ex.x), F(ex.dt), dt_bias, dt_softplus, dt_limit_lo, dt_limit_hi,
                              A, F(ex.B), F(ex.C), D, z ? F(ex.z) : nullptr, initial_states,
                              seq_idx, F(ex.dout), batch, seqlen, nheads, headdim, dstate,
                              ngroups, chunk_size, F(ex.dx), F(ex.ddt), d_dt_bias, dA, F(ex.dB),
                              F(ex.dC), dD, z ? F(ex.dz) : nullptr, d_initial_states, workspace,
                              base, stream);
  if (rc != SSD_OK) return rc;
  down(ex.dx, xs, dx);
  down(ex.ddt, ts, ddt);
  down(ex.dB, bs, dB);
  down(ex.dC, bs, dC);
  if (z) down(ex.dz, xs, dz);
  e = cudaGetLastError();
  if (e != cudaSuccess) {
    char m[200];
    snprintf(m, sizeof(m), "ssd_scan_bwd_ex launch: %s", cudaGetErrorString(e));
    return bfail(SSD_ERR_CUDA, m);
  }
  return SSD_OK;
}

}  // extern "C"
