// The four stages of the SSD chunked-scan forward as CUDA-core (SIMT) kernels
// for sm_103a, templated on the element type (float or bf16) of x/B/C/z/out.
// Accumulation, cumsums and states are fp32; there is no TF32 anywhere.
//
// Stage formulas (chunk c of length Q starting at token t0, head h, group
// g = h / (nheads/ngroups), cs = inclusive cumsum of dt*A inside the chunk):
//   1 dt_cumsum     dt = clamp(softplus(dt_raw + dt_bias)); cs
//   2 chunk_state   S_c[p,n]  = sum_j w_j x_j[p] B_j[n],  w_j = exp(cs_last-cs_j) dt_j
//   3 state_passing H_c = keep_c exp(cs_last) H_{c-1} + S_c
//   4 chunk_scan    y_i = sum_{j<=i} exp(cs_i-cs_j)(C_i.B_j) dt_j x_j   (j < i: strict)
//                         + keep_i exp(cs_i) H_{c-1} C_i + D x_i, then * silu(z_i)
// The recurrence these implement is h_t = exp(dt_t A) h_{t-1} + dt_t x_t B_t^T,
// y_t = h_t C_t + D x_t; chunking it this way is the SSD "chunked scan" of
// mamba_chunk_scan_combined that fla-org/flash-linear-attention PR #49 compares
// with its chunked simple-GLA kernel.
#include <type_traits>

#include "ssd_common.cuh"

namespace ssd {

// ---------------------------------------------------------------------------
// Stage 1: dt preprocessing + per-chunk cumsum of dt*A (+ segment counts)
// grid (nchunks, batch, ceil(nheads/32)), 256 threads: each block takes 32
// heads of one chunk through a [Q][32] shared tile, so that the dt loads are
// coalesced along heads, and each warp then scans one head along the chunk.
// The head-block-0 blocks also write the chunk's segment counts.
// ---------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(256) dt_cumsum_kernel(
    const T* __restrict__ dt, const float* __restrict__ dt_bias, int softplus, float lo,
    float hi, int do_clamp, const float* __restrict__ A, const int32_t* __restrict__ seq_idx,
    Dims d, float* __restrict__ dt_out, float* __restrict__ cs_out, int32_t* __restrict__ seg) {
  __shared__ float tile[256][33];
  __shared__ int warp_tot[8];
  const int c = blockIdx.x, b = blockIdx.y, hb = blockIdx.z;
  const int Q = d.chunk, H = d.nheads;
  const int64_t t0 = (int64_t)c * Q;
  const int n = (int)min((int64_t)Q, d.seqlen - t0);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (seq_idx != nullptr && seg != nullptr && hb == 0) {
    // inclusive count of resets over the chunk; position t0 compares with t0-1
    int flag = 0;
    if (tid < n) {
      const int64_t t = t0 + tid;
      if (t >= 1) flag = seq_idx[b * d.seqlen + t] != seq_idx[b * d.seqlen + t - 1];
    }
    int v = flag;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int o = __shfl_up_sync(0xffffffffu, v, off);
      if (lane >= off) v += o;
    }
    if (lane == 31) warp_tot[warp] = v;
    __syncthreads();
    int pre = 0;
    for (int w = 0; w < warp; ++w) pre += warp_tot[w];
    if (tid < Q) seg[((int64_t)b * d.nchunks + c) * Q + tid] = v + pre;
  }

  const int E = Q >= 32 ? Q / 32 : 1;  // consecutive positions per lane
  const int lq = __ffs(Q) - 1;          // Q is a power of two
  for (int hg = hb * 32; hg < min(H, hb * 32 + 32); hg += 32) {
    const int hw = min(32, H - hg);
    // four positions per thread at a time: their loads first, then the arithmetic
    for (int i0 = tid; i0 < Q * 32; i0 += 4 * 256) {
      float raw[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = i0 + 256 * u, t = idx >> 5, j = idx & 31;
        raw[u] = (idx < Q * 32 && t < n && j < hw) ? to_f(dt[toff(d.sdt, b, t0 + t) + hg + j])
                                                    : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int idx = i0 + 256 * u, t = idx >> 5, j = idx & 31;
        if (idx >= Q * 32) break;
        float v = raw[u];
        if (t < n && j < hw) {
          if (dt_bias) v += dt_bias[hg + j];
          if (softplus) v = v <= 20.f ? log1pf(__expf(v)) : v;
          if (do_clamp) v = fminf(fmaxf(v, lo), hi);
        }
        tile[t][j] = v;
      }
    }
    __syncthreads();
    // the outputs leave with consecutive threads on consecutive positions of
    // one head's row ([B, H, nc, Q]): dt first, then the cumsum, which the
    // scans below write over the tile
    auto row_of = [&](int j) { return (((int64_t)b * H + hg + j) * d.nchunks + c) << lq; };
#pragma unroll 4
    for (int idx = tid; idx < hw << lq; idx += 256)
      dt_out[row_of(idx >> lq) + (idx & (Q - 1))] = tile[idx & (Q - 1)][idx >> lq];
    __syncthreads();
    for (int j = warp; j < hw; j += 8) {
      const float a = A[hg + j];
      float loc[8];
      float run = 0.f;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e < E) {
          const int t = lane * E + e;
          const float v = t < Q ? tile[t][j] * a : 0.f;
          run += v;
          loc[e] = run;
        }
      }
      float incl = run;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      const float excl = incl - run;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (e < E) {
          const int t = lane * E + e;
          if (t < Q) tile[t][j] = excl + loc[e];
        }
      }
    }
    __syncthreads();
#pragma unroll 4
    for (int idx = tid; idx < hw << lq; idx += 256)
      cs_out[row_of(idx >> lq) + (idx & (Q - 1))] = tile[idx & (Q - 1)][idx >> lq];
    __syncthreads();
  }
}

template <typename T>
cudaError_t launch_dt_cumsum(const T* dt, const float* dt_bias, int softplus, float lo,
                             float hi, int do_clamp, const float* A, const int32_t* seq_idx,
                             const Dims& d, float* dt_out, float* cs, int32_t* seg,
                             cudaStream_t st) {
  dim3 grid(d.nchunks, (unsigned)d.batch, (unsigned)((d.nheads + 31) / 32));
  dt_cumsum_kernel<T><<<grid, 256, 0, st>>>(dt, dt_bias, softplus, lo, hi, do_clamp, A,
                                            seq_idx, d, dt_out, cs, seg);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Stage 2: chunk states.  One block per (batch*chunk, head, n-tile) computes
// a [P x NT] tile of S_c as a 32-token-deep SIMT GEMM; the per-token weight
// w_j is applied to x while it is staged in shared memory.
// ---------------------------------------------------------------------------
template <typename T, int P, int NT>
__global__ void __launch_bounds__(256) chunk_state_kernel(
    const T* __restrict__ x, const T* __restrict__ Bm, const float* __restrict__ dtp,
    const float* __restrict__ cs, const int32_t* __restrict__ seg, Dims d,
    float* __restrict__ states) {
  constexpr int TJ = 32, PA = P / 16, NB = NT / 16;
  __shared__ float xs[TJ][P];
  __shared__ float bs[TJ][NT];
  __shared__ float wj[TJ];
  const int bc = blockIdx.x, h = blockIdx.y, ntile = blockIdx.z;
  const int b = bc / d.nchunks, c = bc % d.nchunks;
  const int g = h / (d.nheads / d.ngroups);
  const int Q = d.chunk;
  const int64_t t0 = (int64_t)c * Q;
  const int n = (int)min((int64_t)Q, d.seqlen - t0);
  const int64_t hc = (((int64_t)b * d.nheads + h) * d.nchunks + c) * Q;
  const float* csp = cs + hc;
  const float* dtc = dtp + hc;
  const float cs_last = csp[Q - 1];
  const int32_t* segp = seg ? seg + ((int64_t)b * d.nchunks + c) * Q : nullptr;
  const int seg_last = segp ? segp[Q - 1] : 0;
  const int tid = threadIdx.x, tp = tid / 16, tn = tid % 16;

  float acc[PA][NB];
#pragma unroll
  for (int a = 0; a < PA; ++a)
#pragma unroll
    for (int q = 0; q < NB; ++q) acc[a][q] = 0.f;

  for (int j0 = 0; j0 < n; j0 += TJ) {
    if (tid < TJ) {
      const int j = j0 + tid;
      float w = 0.f;
      if (j < n && (segp == nullptr || segp[j] == seg_last))
        w = ex2((cs_last - csp[j]) * kLog2e) * dtc[j];
      wj[tid] = w;
    }
    __syncthreads();
    for (int idx = tid; idx < TJ * P; idx += 256) {
      const int jj = idx / P, p = idx % P, j = j0 + jj;
      float v = 0.f;
      if (j < n) v = to_f(x[toff(d.sx, b, t0 + j) + (int64_t)(h / d.xrep) * P + p]) * wj[jj];
      xs[jj][p] = v;
    }
    for (int idx = tid; idx < TJ * NT; idx += 256) {
      const int jj = idx / NT, nn = idx % NT, j = j0 + jj;
      float v = 0.f;
      if (j < n)
        v = to_f(Bm[toff(d.sB, b, t0 + j) + (int64_t)g * d.dstate + ntile * NT + nn]);
      bs[jj][nn] = v;
    }
    __syncthreads();
#pragma unroll 4
    for (int jj = 0; jj < TJ; ++jj) {
      float xv[PA], bv[NB];
#pragma unroll
      for (int a = 0; a < PA; ++a) xv[a] = xs[jj][tp + 16 * a];
#pragma unroll
      for (int q = 0; q < NB; ++q) bv[q] = bs[jj][tn + 16 * q];
#pragma unroll
      for (int a = 0; a < PA; ++a)
#pragma unroll
        for (int q = 0; q < NB; ++q) acc[a][q] = fmaf(xv[a], bv[q], acc[a][q]);
    }
    __syncthreads();
  }
  float* sp = states + (((int64_t)b * d.nchunks + c) * d.nheads + h) * (int64_t)P * d.dstate +
              ntile * NT;
#pragma unroll
  for (int a = 0; a < PA; ++a)
#pragma unroll
    for (int q = 0; q < NB; ++q) sp[(int64_t)(tp + 16 * a) * d.dstate + tn + 16 * q] = acc[a][q];
}

template <typename T, int P>
static cudaError_t chunk_state_p(const T* x, const T* B, const float* dtp, const float* cs,
                                 const int32_t* seg, const Dims& d, float* states,
                                 cudaStream_t st) {
  const int NT = d.dstate % 64 == 0 ? 64 : (d.dstate % 32 == 0 ? 32 : 16);
  dim3 grid((unsigned)(d.batch * d.nchunks), d.nheads, d.dstate / NT);
  if (NT == 64)
    chunk_state_kernel<T, P, 64><<<grid, 256, 0, st>>>(x, B, dtp, cs, seg, d, states);
  else if (NT == 32)
    chunk_state_kernel<T, P, 32><<<grid, 256, 0, st>>>(x, B, dtp, cs, seg, d, states);
  else
    chunk_state_kernel<T, P, 16><<<grid, 256, 0, st>>>(x, B, dtp, cs, seg, d, states);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_chunk_state(const T* x, const T* B, const float* dtp, const float* cs,
                               const int32_t* seg, const Dims& d, float* states,
                               cudaStream_t st) {
  if constexpr (std::is_same<T, float>::value) {
    if (chunk_state_tc32_fits(x, B, d))
      return launch_chunk_state_tc32(x, B, dtp, cs, seg, d, states, st);
  }
  switch (d.headdim) {
    case 16: return chunk_state_p<T, 16>(x, B, dtp, cs, seg, d, states, st);
    case 32: return chunk_state_p<T, 32>(x, B, dtp, cs, seg, d, states, st);
    case 64: return chunk_state_p<T, 64>(x, B, dtp, cs, seg, d, states, st);
    case 128: return chunk_state_p<T, 128>(x, B, dtp, cs, seg, d, states, st);
  }
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Stage 3: state passing.  Sequential over chunks, parallel over
// batch x head x (headdim*dstate); each thread owns 4 consecutive state
// elements (float4, coalesced) and rewrites S_c in place with H_{c-1}.
// Loads of the next chunks are issued ahead to keep several in flight.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) state_passing_kernel(
    float* __restrict__ states, const float* __restrict__ cs, const int32_t* __restrict__ seg,
    const float* __restrict__ init, float* __restrict__ final_states, Dims d) {
  const int64_t PN = (int64_t)d.headdim * d.dstate;
  const int64_t e = ((int64_t)blockIdx.x * 256 + threadIdx.x) * 4;
  if (e >= PN) return;
  const int h = blockIdx.y, b = blockIdx.z, Q = d.chunk, nc = d.nchunks;
  float4 hc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (init) hc = *reinterpret_cast<const float4*>(init + ((int64_t)b * d.nheads + h) * PN + e);
  const int64_t cstride = (int64_t)d.nheads * PN;
  float* sp = states + ((int64_t)b * nc * d.nheads + h) * PN + e;
  const float* csp = cs + ((int64_t)b * d.nheads + h) * nc * Q + (Q - 1);
  const int32_t* segp = seg ? seg + (int64_t)b * nc * Q + (Q - 1) : nullptr;
  constexpr int AHEAD = 4;
  float4 buf[AHEAD];
#pragma unroll
  for (int k = 0; k < AHEAD; ++k)
    if (k < nc) buf[k] = *reinterpret_cast<const float4*>(sp + k * cstride);
  for (int c0 = 0; c0 < nc; c0 += AHEAD) {
#pragma unroll
    for (int k = 0; k < AHEAD; ++k) {
      const int c = c0 + k;
      if (c < nc) {
        const float4 s = buf[k];
        if (c + AHEAD < nc) buf[k] = *reinterpret_cast<const float4*>(sp + (c + AHEAD) * cstride);
        *reinterpret_cast<float4*>(sp + c * cstride) = hc;
        const bool keep = segp == nullptr || segp[(int64_t)c * Q] == 0;
        const float dec = keep ? ex2(csp[(int64_t)c * Q] * kLog2e) : 0.f;
        hc.x = fmaf(dec, hc.x, s.x);
        hc.y = fmaf(dec, hc.y, s.y);
        hc.z = fmaf(dec, hc.z, s.z);
        hc.w = fmaf(dec, hc.w, s.w);
      }
    }
  }
  if (final_states)
    *reinterpret_cast<float4*>(final_states + ((int64_t)b * d.nheads + h) * PN + e) = hc;
}

cudaError_t launch_state_passing(float* states, const float* cs, const int32_t* seg,
                                 const float* init, float* final_states, const Dims& d,
                                 cudaStream_t st) {
  const int64_t PN = (int64_t)d.headdim * d.dstate;
  dim3 grid((unsigned)((PN / 4 + 255) / 256), d.nheads, (unsigned)d.batch);
  state_passing_kernel<<<grid, 256, 0, st>>>(states, cs, seg, init, final_states, d);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Stage 4: chunk scan.  One block per (batch*chunk, head, 32-row tile); 256
// threads = 32 rows x 8 column groups, each thread accumulating P/8 outputs
// of its row.  Inter-chunk term first (C_i . H_{c-1}, scaled by exp(cs_i)),
// then the causal intra-chunk term one 32-token tile at a time, then the
// D skip and the silu(z) gate.
// ---------------------------------------------------------------------------
template <typename T, int P>
__global__ void __launch_bounds__(256) chunk_scan_kernel(
    const T* __restrict__ x, const T* __restrict__ Bm, const T* __restrict__ Cm,
    const float* __restrict__ dtp, const float* __restrict__ cs,
    const int32_t* __restrict__ seg, const float* __restrict__ prev,
    const float* __restrict__ D, const T* __restrict__ z, Dims d, T* __restrict__ out,
    int strict) {
  constexpr int TI = 32, TJ = 32, NTL = 16, KP = P / 8;
  extern __shared__ float smem[];
  const int N = d.dstate, NP1 = N + 1;
  float* Cs = smem;                   // [TI][N+1]
  float* Bs = Cs + TI * NP1;          // [TJ][N+1]
  float* Hs = Bs + TJ * NP1;          // [P][NTL+1]
  float* xs = Hs + P * (NTL + 1);     // [TJ][P]
  float* Ms = xs + TJ * P;            // [TI][TJ+1]
  float* cs_i = Ms + TI * (TJ + 1);   // [TI]
  float* cs_j = cs_i + TI;            // [TJ]
  int* sg_i = reinterpret_cast<int*>(cs_j + TJ);
  int* sg_j = sg_i + TI;

  const int bc = blockIdx.x, h = blockIdx.y, rt = blockIdx.z;
  const int b = bc / d.nchunks, c = bc % d.nchunks;
  const int g = h / (d.nheads / d.ngroups);
  const int Q = d.chunk;
  const int64_t t0 = (int64_t)c * Q;
  const int n = (int)min((int64_t)Q, d.seqlen - t0);
  const int i0 = rt * TI;
  if (i0 >= n) return;  // whole block past the end of a short last chunk
  const int64_t hc = (((int64_t)b * d.nheads + h) * d.nchunks + c) * Q;
  const float* csp = cs + hc;
  const float* dtc = dtp + hc;
  const int32_t* segp = seg ? seg + ((int64_t)b * d.nchunks + c) * Q : nullptr;
  const int tid = threadIdx.x, r = tid / 8, cg = tid % 8;
  const int64_t rowBC = (int64_t)b * d.seqlen + t0;  // token row of the chunk start

  for (int idx = tid; idx < TI * N; idx += 256) {
    const int ii = idx / N, nn = idx % N, i = i0 + ii;
    Cs[ii * NP1 + nn] = i < n ? to_f(Cm[toff(d.sC, b, t0 + i) + (int64_t)g * N + nn]) : 0.f;
  }
  if (tid < TI) {
    const int i = min(i0 + tid, Q - 1);
    cs_i[tid] = csp[i];
    sg_i[tid] = segp ? segp[i] : 0;
  }
  __syncthreads();

  float acc[KP];
#pragma unroll
  for (int k = 0; k < KP; ++k) acc[k] = 0.f;

  // inter-chunk term: C_i . H_{c-1}
  const float* Hp = prev + (((int64_t)b * d.nchunks + c) * d.nheads + h) * (int64_t)P * N;
  for (int n0 = 0; n0 < N; n0 += NTL) {
    for (int idx = tid; idx < P * NTL; idx += 256) {
      const int p = idx / NTL, nn = idx % NTL;
      Hs[p * (NTL + 1) + nn] = Hp[(int64_t)p * N + n0 + nn];
    }
    __syncthreads();
#pragma unroll
    for (int nn = 0; nn < NTL; ++nn) {
      const float cv = Cs[r * NP1 + n0 + nn];
#pragma unroll
      for (int k = 0; k < KP; ++k) acc[k] = fmaf(cv, Hs[(cg + 8 * k) * (NTL + 1) + nn], acc[k]);
    }
    __syncthreads();
  }
  {
    const float sc = sg_i[r] == 0 ? ex2(cs_i[r] * kLog2e) : 0.f;
#pragma unroll
    for (int k = 0; k < KP; ++k) acc[k] *= sc;
  }

  // intra-chunk causal term
  const int irow = i0 + r;
  for (int jt = 0; jt <= rt; ++jt) {
    const int j0 = jt * TJ;
    for (int idx = tid; idx < TJ * N; idx += 256) {
      const int jj = idx / N, nn = idx % N, j = j0 + jj;
      Bs[jj * NP1 + nn] = j < n ? to_f(Bm[toff(d.sB, b, t0 + j) + (int64_t)g * N + nn]) : 0.f;
    }
    for (int idx = tid; idx < TJ * P; idx += 256) {
      const int jj = idx / P, p = idx % P, j = j0 + jj;
      xs[jj * P + p] =
          j < n ? to_f(x[toff(d.sx, b, t0 + j) + (int64_t)(h / d.xrep) * P + p]) * dtc[j] : 0.f;
    }
    if (tid < TJ) {
      const int j = min(j0 + tid, Q - 1);
      cs_j[tid] = csp[j];
      sg_j[tid] = segp ? segp[j] : 0;
    }
    __syncthreads();
    float s[4];
#pragma unroll
    for (int m = 0; m < 4; ++m) s[m] = 0.f;
    for (int nn = 0; nn < N; ++nn) {
      const float cv = Cs[r * NP1 + nn];
#pragma unroll
      for (int m = 0; m < 4; ++m) s[m] = fmaf(cv, Bs[(cg + 8 * m) * NP1 + nn], s[m]);
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const int jj = cg + 8 * m, j = j0 + jj;
      const bool valid = j + strict <= irow && j < n && sg_j[jj] == sg_i[r];
      Ms[r * (TJ + 1) + jj] = valid ? s[m] * ex2((cs_i[r] - cs_j[jj]) * kLog2e) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int jj = 0; jj < TJ; ++jj) {
      const float mv = Ms[r * (TJ + 1) + jj];
#pragma unroll
      for (int k = 0; k < KP; ++k) acc[k] = fmaf(mv, xs[jj * P + cg + 8 * k], acc[k]);
    }
    __syncthreads();
  }

  if (irow < n) {
    const int64_t base = ((rowBC + irow) * d.nheads + h) * P;   // out (dense)
    const int64_t xbase = toff(d.sx, b, t0 + irow) + (int64_t)(h / d.xrep) * P;
    const int64_t zbase = toff(d.sz, b, t0 + irow) + (int64_t)h * P;
    const float Dh = D ? D[h] : 0.f;
#pragma unroll
    for (int k = 0; k < KP; ++k) {
      const int p = cg + 8 * k;
      float y = acc[k];
      if (D) y = fmaf(Dh, to_f(x[xbase + p]), y);
      if (z) {
        const float zz = to_f(z[zbase + p]);
        y *= zz / (1.f + __expf(-zz));
      }
      out[base + p] = from_f<T>(y);
    }
  }
}

template <typename T, int P>
static cudaError_t chunk_scan_p(const T* x, const T* B, const T* C, const float* dtp,
                                const float* cs, const int32_t* seg, const float* prev,
                                const float* D, const T* z, const Dims& d, T* out,
                                cudaStream_t st, int strict) {
  constexpr int TI = 32, TJ = 32, NTL = 16;
  const int NP1 = d.dstate + 1;
  const size_t smem = sizeof(float) * ((size_t)TI * NP1 + (size_t)TJ * NP1 + (size_t)P * (NTL + 1) +
                                       (size_t)TJ * P + (size_t)TI * (TJ + 1) + TI + TJ) +
                      sizeof(int) * (TI + TJ);
  auto kern = chunk_scan_kernel<T, P>;
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
  }
  dim3 grid((unsigned)(d.batch * d.nchunks), d.nheads, (d.chunk + TI - 1) / TI);
  kern<<<grid, 256, smem, st>>>(x, B, C, dtp, cs, seg, prev, D, z, d, out, strict);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_chunk_scan(const T* x, const T* B, const T* C, const float* dtp,
                              const float* cs, const int32_t* seg, const float* prev,
                              const float* D, const T* z, const Dims& d, T* out,
                              cudaStream_t st, int strict) {
  if constexpr (std::is_same<T, float>::value) {
    if (chunk_scan_tc32_fits(x, B, C, z, d))
      return launch_chunk_scan_tc32(x, B, C, dtp, cs, seg, prev, D, z, d, out, st, strict);
  }
  switch (d.headdim) {
    case 16: return chunk_scan_p<T, 16>(x, B, C, dtp, cs, seg, prev, D, z, d, out, st,
                                             strict);
    case 32: return chunk_scan_p<T, 32>(x, B, C, dtp, cs, seg, prev, D, z, d, out, st,
                                             strict);
    case 64: return chunk_scan_p<T, 64>(x, B, C, dtp, cs, seg, prev, D, z, d, out, st,
                                             strict);
    case 128: return chunk_scan_p<T, 128>(x, B, C, dtp, cs, seg, prev, D, z, d, out, st,
                                             strict);
  }
  return cudaErrorInvalidValue;
}

// explicit instantiations for the two supported element types
#define SSD_INSTANTIATE(T)                                                                      \
  template cudaError_t launch_dt_cumsum<T>(const T*, const float*, int, float, float, int,      \
                                           const float*, const int32_t*, const Dims&, float*,   \
                                           float*, int32_t*, cudaStream_t);                      \
  template cudaError_t launch_chunk_state<T>(const T*, const T*, const float*, const float*,    \
                                             const int32_t*, const Dims&, float*, cudaStream_t); \
  template cudaError_t launch_chunk_scan<T>(const T*, const T*, const T*, const float*,         \
                                            const float*, const int32_t*, const float*,         \
                                            const float*, const T*, const Dims&, T*, cudaStream_t, \
                                            int);
SSD_INSTANTIATE(float)
SSD_INSTANTIATE(__nv_bfloat16)

}  // namespace ssd
