// fp32 stages 2 and 4 of the SSD chunked scan (chunk_state, chunk_scan) on
// the tensor cores, for 128-token chunks.  tcgen05.mma kind::tf32 reads
// only the top 19 bits of an fp32 operand, so each operand v is split into
// hi = v rounded to tf32 and lo = v - hi (exact in fp32), and every product
// takes three MMAs into the same fp32 TMEM accumulator:
//   A B ~ A_hi B_hi + A_hi B_lo + A_lo B_hi
// (the dropped A_lo B_lo is below 2^-22 of the product), i.e. about fp32
// accuracy at tensor-core rate.  The formulas are those of the SIMT stages
// (ssd_simt.cu), chunk c of Q = 128 tokens from t0, head h, group g:
//   chunk_state  S_c[p,n] = sum_j w_j x_j[p] B_j[n],  w_j = exp(cs_last - cs_j) dt_j
//   chunk_scan   y_i = sum_{j<=i} exp(cs_i - cs_j) (C_i . B_j) dt_j x_j
//                      + keep_i exp(cs_i) C_i . H_{c-1} + D x_i,  then * silu(z_i)
// Operands are split and written K-major into 64-byte-swizzled shared
// tiles by the CUDA cores (transposed where the token index is the K
// dimension), one 16-element K slice at a time into two alternating
// buffers, so that a slice is staged while the previous one's MMAs run; one
// thread issues the MMAs.  chunk_scan runs C B^T into TMEM (K = dstate)
// unless it is given C B^T computed once per group (cb_tc32_kernel), the
// inter-chunk term (e^cs C) H^T into the output accumulator (K = dstate),
// then the decay-masked matrix M = (C B^T) o L o dt, built by the CUDA cores,
// times x (K = tokens).  Every mbarrier wait is bounded by the global timer
// and records a status bit instead of hanging.
#include <stdio.h>
#include <stdlib.h>

#include "ssd_common.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace tc32 {

__device__ int g_status32;

constexpr int kQ = 128;                       // tokens per chunk = MMA rows
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s (the default wait limit)
constexpr int kErrWait = 8;                   // status bit of a timed-out wait

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, uint64_t wait_ns) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (gtimer() - t0 > wait_ns) {
      atomicOr(&g_status32, kErrWait);
      return false;
    }
  }
  return true;
}

// Operand tiles hold K slices of 16 fp32 (64-byte rows) with the 64-byte
// swizzle: 16-byte chunk c of row r sits at chunk c ^ ((r >> 1) & 3).  A
// split tile of R rows keeps the hi rows first and the lo rows after them.
constexpr int kK = 16;   // K elements per slice

__device__ __forceinline__ uint32_t off16(uint32_t row, uint32_t k) {   // k < 16
  return row * 64u + ((((k >> 2) ^ ((row >> 1) & 3u)) << 4) | ((k & 3u) << 2));
}

__device__ __forceinline__ void split(float v, float& hi, float& lo) {
  hi = __uint_as_float((__float_as_uint(v) + 0x1000u) & 0xFFFFE000u);   // nearest tf32
  lo = v - hi;
}

__device__ __forceinline__ void put1(unsigned char* t, int rows, int r, int k, float v) {
  float hi, lo;
  split(v, hi, lo);
  const uint32_t o = off16(r, k);
  *reinterpret_cast<float*>(t + o) = hi;
  *reinterpret_cast<float*>(t + rows * 64 + o) = lo;
}
// four consecutive k (k % 4 == 0) of row r
__device__ __forceinline__ void put4(unsigned char* t, int rows, int r, int k, float4 v) {
  float4 hi, lo;
  split(v.x, hi.x, lo.x);
  split(v.y, hi.y, lo.y);
  split(v.z, hi.z, lo.z);
  split(v.w, hi.w, lo.w);
  const uint32_t o = off16(r, k);
  *reinterpret_cast<float4*>(t + o) = hi;
  *reinterpret_cast<float4*>(t + rows * 64 + o) = lo;
}

__device__ __forceinline__ float4 ld4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}
__device__ __forceinline__ float4 scale4(float4 v, float s) {
  return make_float4(v.x * s, v.y * s, v.z * s, v.w * s);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::tf32: tf32 A and B (K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4) | (2u << 7) | (2u << 10) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Shared-memory descriptor of a K-major tile with the 64-byte swizzle:
// 8-row groups of 64-byte rows 512 bytes apart (SBO), one swizzle atom wide
// in K (LBO unused), base 512-byte aligned.
__device__ __forceinline__ uint64_t sdesc_sw64(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;    // LBO (16 bytes, unused)
  d |= static_cast<uint64_t>(512u >> 4) << 32;
  d |= 1ull << 46;                         // descriptor version used by tcgen05
  d |= 4ull << 61;                         // 64-byte swizzle
  return d;
}

// D (+)= A B^T over one 16-wide K slice of split tiles (3 x 2 MMAs).
// a: 128 rows, b: nb rows; the first MMA overwrites D unless acc.
__device__ __forceinline__ void mma_slice(uint32_t d, const unsigned char* a,
                                          const unsigned char* b, int nb, uint32_t idesc,
                                          bool acc) {
  const uint64_t ah = sdesc_sw64(tc::smem_u32(a));
  const uint64_t al = sdesc_sw64(tc::smem_u32(a + kQ * 64));
  const uint64_t bh = sdesc_sw64(tc::smem_u32(b));
  const uint64_t bl = sdesc_sw64(tc::smem_u32(b + nb * 64));
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const uint64_t o = static_cast<uint64_t>(k * 2);   // 32 bytes, in 16-byte units
    mma_tf32(d, ah + o, bh + o, idesc, (acc || k > 0) ? 1u : 0u);
    mma_tf32(d, ah + o, bl + o, idesc, 1u);
    mma_tf32(d, al + o, bh + o, idesc, 1u);
  }
}

__device__ __forceinline__ unsigned char* aligned_smem(unsigned char* raw) {
  return raw + ((1024u - (tc::smem_u32(raw) & 1023u)) & 1023u);
}

// Two buffers of split tiles, 32 KB each (A: 128 rows, B: up to 128 rows,
// hi and lo, 64-byte rows).  Slice s fills buffer s % 2 while the MMAs of
// slice s - 1 read the other one; before the fill, the MMAs of slice s - 2
// (the buffer's previous contents) must be complete.
constexpr int kBuf = 2 * kQ * 64 * 2;   // bytes per buffer

// The pipeline both kernels run: slice s waits for its buffer, stores its
// operands (from registers loaded two slices earlier) and loads those of
// slice s + 2, then, once every thread has stored, one thread issues the
// slice's MMAs and commits them to the buffer's mbarrier.  Returns false if a
// bounded wait gave up (uniform over the CTA).
// (`Limits`: the wait limit, and the test-only option under which the first
// CTA leaves its first slice uncommitted, so that a wait runs out.)
struct Limits {
  uint64_t wait_ns;
  int stall;
};

template <typename Store, typename Load, typename Issue>
__device__ __forceinline__ bool pipeline_step(int s, int nS, uint64_t* bars, int tid,
                                             int& ok_all, const Limits& lim, Store&& store,
                                             Load&& load, Issue&& issue) {
  bool ok = true;
  if (s >= 2) ok = wait_phase(&bars[s & 1], ((s - 2) >> 1) & 1, lim.wait_ns);
  tc::fence_after_sync();
  if (ok) store(s);
  if (s + 2 < nS) load(s + 2);
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  if (!ok) ok_all = 0;
  if (!__syncthreads_and(ok)) return false;
  tc::fence_after_sync();
  if (tid == 0) {
    issue(s);
    if (!(lim.stall && s == 0 && blockIdx.x == 0 && blockIdx.y == 0)) tc::mma_commit(&bars[s & 1]);
  }
  return true;
}

// Waits for the last slice's MMAs (so every earlier one) before the
// accumulators are read or the TMEM is freed.
__device__ __forceinline__ bool pipeline_drain(int nS, uint64_t* bars, int& ok_all,
                                               const Limits& lim) {
  bool ok = true;
  if (nS > 0) ok = wait_phase(&bars[(nS - 1) & 1], ((nS - 1) >> 1) & 1, lim.wait_ns);
  tc::fence_after_sync();
  if (!ok) ok_all = 0;
  return __syncthreads_and(ok) != 0;
}

// ---------------------------------------------------------------------------
// A per-group operand Y [batch, seqlen, groups, 128] (B, or the reversed C)
// written once as chunk_state's A tiles: for every (batch x chunk, group)
// and 16-token slice, the 128 x 16 transpose (row = Y's feature, K = token)
// split into hi and lo and laid out as the shared tile (64-byte swizzle),
// 16 KB per slice, so that chunk_state copies it instead of staging it for
// every head.  One CTA per (batch x chunk, group, slice), 256 threads:
// thread (row = tid % 128, tokens 8 (tid / 128) .. + 7).
// ---------------------------------------------------------------------------
constexpr int kTileFloats = kQ * kK * 2;   // floats per split slice (hi + lo)

__global__ void __launch_bounds__(256) group_tiles_kernel(const float* __restrict__ Y,
                                                          TokStride sY, int groups,
                                                          int64_t seqlen, int nchunks,
                                                          float* __restrict__ T) {
  const int bc = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int64_t b = bc / nchunks;
  const int c = bc % nchunks;
  const int row = threadIdx.x % kQ, k0 = 8 * (threadIdx.x / kQ);
  const int64_t t0 = (int64_t)c * kQ + kK * s;
  unsigned char* tile = reinterpret_cast<unsigned char*>(
      T + (((int64_t)bc * groups + g) * (kQ / kK) + s) * kTileFloats);
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const int k = k0 + u;
    const int64_t t = t0 + k;
    const float v = t < seqlen ? Y[toff(sY, b, t) + (int64_t)g * kQ + row] : 0.f;
    put1(tile, kQ, row, k, v);
  }
}

// ---------------------------------------------------------------------------
// chunk_state: one CTA per (batch x chunk, head), 256 threads.  The MMA rows
// are the 128-wide one of headdim / dstate: with dstate 128 the transposed
// state S^T = B^T (w o x) (rows n), else S = (w o x)^T B (rows p).  K = the
// chunk's tokens, 16-token slices; both operands are staged transposed
// (16 lanes on the tokens, the other half-warp on the next row quad).
// ---------------------------------------------------------------------------
// kG: the 128-row operand is per group (B when dstate is 128; x, read
// through xrep, when headdim is 128) and comes pre-split from Tg
// (group_tiles_kernel); the weights w_j then go on the other, per-head
// operand (the sum over j of w_j x_j B_j^T does not care which factor
// carries them), the only one staged here.
// (three CTAs per SM, as its shared memory allows: up to 85 registers)
template <int P, int N, bool kG>
__global__ void __launch_bounds__(256, 3) chunk_state_tc32_kernel(
    const float* __restrict__ x, const float* __restrict__ Bm, const float* __restrict__ dtp,
    const float* __restrict__ cs, const int32_t* __restrict__ seg, Dims d,
    float* __restrict__ states, Limits lim, const float* __restrict__ Tg) {
  constexpr bool kT = (N == 128);
  constexpr int NR = kT ? P : N;   // MMA N: the other dimension
  constexpr int XQ = P / 64, BQ = N / 64;   // row quads per thread and slice (16 per warp)
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = aligned_smem(smem_raw);
  __shared__ float wsh[kQ];
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_base;
  __shared__ int ok_all;

  const int bc = blockIdx.x, h = blockIdx.y;
  const int b = bc / d.nchunks, c = bc % d.nchunks;
  const int g = h / (d.nheads / d.ngroups);
  const int64_t t0 = (int64_t)c * kQ;
  const int n = (int)min((int64_t)kQ, d.seqlen - t0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t hc = (((int64_t)b * d.nheads + h) * d.nchunks + c) * kQ;
  if (tid < kQ) {
    const int32_t* sp = seg ? seg + ((int64_t)b * d.nchunks + c) * kQ : nullptr;
    float w = 0.f;
    if (tid < n && (sp == nullptr || sp[tid] == sp[kQ - 1]))
      w = ex2((cs[hc + kQ - 1] - cs[hc + tid]) * kLog2e) * dtp[hc + tid];
    wsh[tid] = w;
  }
  if (tid == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::mbar_fence_init();
    ok_all = 1;
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 128);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  constexpr uint32_t idesc = idesc_tf32(kQ, NR);
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* xh = x + (int64_t)(h / d.xrep) * P;
  const float* bg = Bm + (int64_t)g * N;
  const int jl = lane & 15, qh = lane >> 4;   // token in the slice, row-quad half
  // tiles of buffer u: A (128 rows) then B (NR rows)
  auto tA = [&](int u) { return base + u * kBuf; };
  auto tB = [&](int u) { return base + u * kBuf + kQ * 128; };

  const int nS = (n + kK - 1) / kK;
  // two register sets: slice s + 2 loads while slice s is stored / multiplied
  // (with the weight w of this lane's token, read from shared memory then)
  float4 rx0[XQ], rb0[BQ], rx1[XQ], rb1[BQ];
  float w0 = 0.f, w1 = 0.f;
  auto load_into = [&](int s, float4(&rx)[XQ], float4(&rb)[BQ], float& w) {
    const int j = kK * s + jl;
    const bool tv = j < n;
    w = tv ? wsh[j] : 0.f;
    const int64_t tx = toff(d.sx, b, t0 + (tv ? j : 0)), tb = toff(d.sB, b, t0 + (tv ? j : 0));
#pragma unroll
    for (int u = 0; u < XQ; ++u) rx[u] = tv ? ld4(xh + tx + 4 * (2 * warp + qh + 16 * u)) : zero4;
#pragma unroll
    for (int u = 0; u < BQ; ++u) rb[u] = tv ? ld4(bg + tb + 4 * (2 * warp + qh + 16 * u)) : zero4;
  };
  auto store_from = [&](int s, const float4(&rx)[XQ], const float4(&rb)[BQ], float wj) {
    unsigned char* tX = kT ? tB(s & 1) : tA(s & 1);    // (w o x)^T: P rows
    unsigned char* tBt = kT ? tA(s & 1) : tB(s & 1);   // B^T: N rows
#pragma unroll
    for (int u = 0; u < XQ; ++u) {
      const int r = 4 * (2 * warp + qh + 16 * u);
      put1(tX, P, r, jl, rx[u].x * wj);
      put1(tX, P, r + 1, jl, rx[u].y * wj);
      put1(tX, P, r + 2, jl, rx[u].z * wj);
      put1(tX, P, r + 3, jl, rx[u].w * wj);
    }
#pragma unroll
    for (int u = 0; u < BQ; ++u) {
      const int r = 4 * (2 * warp + qh + 16 * u);
      put1(tBt, N, r, jl, rb[u].x);
      put1(tBt, N, r + 1, jl, rb[u].y);
      put1(tBt, N, r + 2, jl, rb[u].z);
      put1(tBt, N, r + 3, jl, rb[u].w);
    }
  };
  auto issue = [&](int s) { mma_slice(tmem, tA(s & 1), tB(s & 1), NR, idesc, s > 0); };

  // kG: the tile copy (four float4 per thread and slice) and the per-head
  // operand, weighted
  constexpr int VQ = kT ? XQ : BQ, VR = kT ? P : N;
  const float* tg = nullptr;
  if (kG) {
    const int tgroups = kT ? d.ngroups : d.nheads / d.xrep;
    const int gi = kT ? g : h / d.xrep;
    tg = Tg + ((int64_t)bc * tgroups + gi) * (kQ / kK) * kTileFloats;
  }
  float4 rt0[4], rv0[VQ], rt1[4], rv1[VQ];
  auto gload_into = [&](int s, float4(&rt)[4], float4(&rv)[VQ], float& w) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      rt[u] = ld4(tg + (int64_t)s * kTileFloats + 4 * (tid + 256 * u));
    const int j = kK * s + jl;
    const bool tv = j < n;
    w = tv ? wsh[j] : 0.f;
    const float* src = kT ? xh + toff(d.sx, b, t0 + (tv ? j : 0))
                          : Bm + toff(d.sB, b, t0 + (tv ? j : 0)) + (int64_t)g * N;
#pragma unroll
    for (int u = 0; u < VQ; ++u) rv[u] = tv ? ld4(src + 4 * (2 * warp + qh + 16 * u)) : zero4;
  };
  auto gstore_from = [&](int s, const float4(&rt)[4], const float4(&rv)[VQ], float wj) {
    float4* a = reinterpret_cast<float4*>(tA(s & 1));
#pragma unroll
    for (int u = 0; u < 4; ++u) a[tid + 256 * u] = rt[u];
    unsigned char* bt = tB(s & 1);
#pragma unroll
    for (int u = 0; u < VQ; ++u) {
      const int r = 4 * (2 * warp + qh + 16 * u);
      put1(bt, VR, r, jl, rv[u].x * wj);
      put1(bt, VR, r + 1, jl, rv[u].y * wj);
      put1(bt, VR, r + 2, jl, rv[u].z * wj);
      put1(bt, VR, r + 3, jl, rv[u].w * wj);
    }
  };

  bool run = true;
  if constexpr (kG) {
    gload_into(0, rt0, rv0, w0);
    if (nS > 1) gload_into(1, rt1, rv1, w1);
    for (int s = 0; run && s < nS; s += 2) {
      run = pipeline_step(s, nS, bars, tid, ok_all, lim,
                          [&](int t) { gstore_from(t, rt0, rv0, w0); },
                          [&](int t) { gload_into(t, rt0, rv0, w0); }, issue);
      if (run && s + 1 < nS)
        run = pipeline_step(s + 1, nS, bars, tid, ok_all, lim,
                            [&](int t) { gstore_from(t, rt1, rv1, w1); },
                            [&](int t) { gload_into(t, rt1, rv1, w1); }, issue);
    }
  } else {
    load_into(0, rx0, rb0, w0);
    if (nS > 1) load_into(1, rx1, rb1, w1);
    for (int s = 0; run && s < nS; s += 2) {
      run = pipeline_step(s, nS, bars, tid, ok_all, lim,
                          [&](int t) { store_from(t, rx0, rb0, w0); },
                          [&](int t) { load_into(t, rx0, rb0, w0); }, issue);
      if (run && s + 1 < nS)
        run = pipeline_step(s + 1, nS, bars, tid, ok_all, lim,
                            [&](int t) { store_from(t, rx1, rb1, w1); },
                            [&](int t) { load_into(t, rx1, rb1, w1); }, issue);
    }
  }
  if (run) run = pipeline_drain(nS, bars, ok_all, lim);
  if (run) {
    // each warp: TMEM lane quarter warp % 4, half of the NR columns
    const int q = warp & 3, half = warp >> 2;
    const int row = 32 * q + lane;   // n (kT) or p
    float* sp = states + (((int64_t)b * d.nchunks + c) * d.nheads + h) * (int64_t)P * N;
    float* ys = reinterpret_cast<float*>(base);
#pragma unroll
    for (int c0 = 0; c0 < NR / 2; c0 += 32) {
      uint32_t r[32];
      const int col0 = half * (NR / 2) + c0;
      tc::tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + col0, r);
      tc::tmem_ld_wait_regs(r);
      if (kT) {   // lanes on consecutive n: each store is one 128-byte row piece
#pragma unroll
        for (int u = 0; u < 32; ++u) sp[(int64_t)(col0 + u) * N + row] = __uint_as_float(r[u]);
      } else {    // rows of N + 4 floats in shared memory (over the tiles)
#pragma unroll
        for (int u = 0; u < 32; u += 4)
          *reinterpret_cast<float4*>(ys + row * (N + 4) + col0 + u) =
              make_float4(__uint_as_float(r[u]), __uint_as_float(r[u + 1]),
                          __uint_as_float(r[u + 2]), __uint_as_float(r[u + 3]));
      }
    }
    if (!kT) {   // then out with consecutive threads on consecutive n
      __syncthreads();
      for (int e = tid; e < P * (N / 4); e += 256) {
        const int pr = e / (N / 4), c4 = 4 * (e % (N / 4));
        *reinterpret_cast<float4*>(sp + (int64_t)pr * N + c4) =
            *reinterpret_cast<const float4*>(ys + pr * (N + 4) + c4);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
// chunk_state for two heads at once where the per-group operand is the
// 128-row one and comes pre-split (kG above) and the per-head operand has 64
// rows (headdim 64 with dstate 128, or dstate 64 with headdim 128): the two
// heads' weighted operands stack into one 128-row B tile, so that every MMA
// has N = 128 (about the time of an N = 64 one, for twice the work) and the
// group tile is copied once for both.  One CTA per (batch x chunk, head
// pair), 256 threads; the pair's heads share the per-group operand.
// Accumulator columns 64 e .. 64 e + 63 belong to head h0 + e.
// ---------------------------------------------------------------------------
template <int P, int N>
__global__ void __launch_bounds__(256, 3) chunk_state_pair_tc32_kernel(
    const float* __restrict__ x, const float* __restrict__ Bm, const float* __restrict__ dtp,
    const float* __restrict__ cs, const int32_t* __restrict__ seg, Dims d,
    float* __restrict__ states, Limits lim, const float* __restrict__ Tg) {
  constexpr bool kT = (N == 128);
  static_assert((kT ? P : N) == 64, "two 64-row per-head operands fill the 128-row B tile");
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = aligned_smem(smem_raw);
  __shared__ float wsh[2][kQ];
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_base;
  __shared__ int ok_all;

  const int bc = blockIdx.x, h0 = 2 * blockIdx.y;
  const int b = bc / d.nchunks, c = bc % d.nchunks;
  const int64_t t0 = (int64_t)c * kQ;
  const int n = (int)min((int64_t)kQ, d.seqlen - t0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  {   // thread (head e, position t): the weight w_t of head h0 + e
    const int e = tid / kQ, t = tid % kQ;
    const int64_t hc = (((int64_t)b * d.nheads + h0 + e) * d.nchunks + c) * kQ;
    const int32_t* sp = seg ? seg + ((int64_t)b * d.nchunks + c) * kQ : nullptr;
    float w = 0.f;
    if (t < n && (sp == nullptr || sp[t] == sp[kQ - 1]))
      w = ex2((cs[hc + kQ - 1] - cs[hc + t]) * kLog2e) * dtp[hc + t];
    wsh[e][t] = w;
  }
  if (tid == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::mbar_fence_init();
    ok_all = 1;
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 128);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  constexpr uint32_t idesc = idesc_tf32(kQ, kQ);
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const int hpg = d.nheads / d.ngroups;
  // the per-head operand of head h0 + e at token t: x (kT), else B (whose
  // groups are the heads there)
  auto head_row = [&](int e, int64_t t) -> const float* {
    return kT ? x + toff(d.sx, b, t) + (int64_t)((h0 + e) / d.xrep) * P
              : Bm + toff(d.sB, b, t) + (int64_t)((h0 + e) / hpg) * N;
  };
  const int tgroups = kT ? d.ngroups : d.nheads / d.xrep;
  const int gi = kT ? h0 / hpg : h0 / d.xrep;
  const float* tg = Tg + ((int64_t)bc * tgroups + gi) * (kQ / kK) * kTileFloats;
  const int jl = lane & 15, qh = lane >> 4;   // token in the slice, row-quad half
  const int r0 = 4 * (2 * warp + qh);         // this thread's row quad of a head's 64 rows
  auto tA = [&](int u) { return base + u * kBuf; };
  auto tB = [&](int u) { return base + u * kBuf + kQ * 128; };
  const int nS = (n + kK - 1) / kK;
  // two register sets: slice s + 2 loads while slice s is stored / multiplied
  float4 rt0[4], rv0[2], rt1[4], rv1[2];
  float2 w0 = make_float2(0.f, 0.f), w1 = make_float2(0.f, 0.f);
  auto load_into = [&](int s, float4(&rt)[4], float4(&rv)[2], float2& w) {
#pragma unroll
    for (int u = 0; u < 4; ++u)
      rt[u] = ld4(tg + (int64_t)s * kTileFloats + 4 * (tid + 256 * u));
    const int j = kK * s + jl;
    const bool tv = j < n;
    const int64_t t = t0 + (tv ? j : 0);
    w = tv ? make_float2(wsh[0][j], wsh[1][j]) : make_float2(0.f, 0.f);
    rv[0] = tv ? ld4(head_row(0, t) + r0) : zero4;
    rv[1] = tv ? ld4(head_row(1, t) + r0) : zero4;
  };
  auto store_from = [&](int s, const float4(&rt)[4], const float4(&rv)[2], float2 w) {
    float4* a = reinterpret_cast<float4*>(tA(s & 1));
#pragma unroll
    for (int u = 0; u < 4; ++u) a[tid + 256 * u] = rt[u];
    unsigned char* bt = tB(s & 1);   // head e's rows at 64 e
    put1(bt, kQ, r0, jl, rv[0].x * w.x);
    put1(bt, kQ, r0 + 1, jl, rv[0].y * w.x);
    put1(bt, kQ, r0 + 2, jl, rv[0].z * w.x);
    put1(bt, kQ, r0 + 3, jl, rv[0].w * w.x);
    put1(bt, kQ, 64 + r0, jl, rv[1].x * w.y);
    put1(bt, kQ, 64 + r0 + 1, jl, rv[1].y * w.y);
    put1(bt, kQ, 64 + r0 + 2, jl, rv[1].z * w.y);
    put1(bt, kQ, 64 + r0 + 3, jl, rv[1].w * w.y);
  };
  auto issue = [&](int s) { mma_slice(tmem, tA(s & 1), tB(s & 1), kQ, idesc, s > 0); };

  bool run = true;
  load_into(0, rt0, rv0, w0);
  if (nS > 1) load_into(1, rt1, rv1, w1);
  for (int s = 0; run && s < nS; s += 2) {
    run = pipeline_step(s, nS, bars, tid, ok_all, lim,
                        [&](int t) { store_from(t, rt0, rv0, w0); },
                        [&](int t) { load_into(t, rt0, rv0, w0); }, issue);
    if (run && s + 1 < nS)
      run = pipeline_step(s + 1, nS, bars, tid, ok_all, lim,
                          [&](int t) { store_from(t, rt1, rv1, w1); },
                          [&](int t) { load_into(t, rt1, rv1, w1); }, issue);
  }
  if (run) run = pipeline_drain(nS, bars, ok_all, lim);
  if (run) {
    // each warp: TMEM lane quarter warp % 4, the 64 columns of head h0 + half
    const int q = warp & 3, half = warp >> 2;
    const int row = 32 * q + lane;   // n (kT) or p
    float* sp = states + (((int64_t)b * d.nchunks + c) * d.nheads + h0 + half) * (int64_t)P * N;
    float* ys = reinterpret_cast<float*>(base);
    constexpr int YS = kQ + 4;   // !kT: rows p of both heads' n, 132 floats
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      uint32_t r[32];
      tc::tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + 64 * half + c0, r);
      tc::tmem_ld_wait_regs(r);
      if (kT) {   // S^T of head h0 + half: lanes on consecutive n
#pragma unroll
        for (int u = 0; u < 32; ++u) sp[(int64_t)(c0 + u) * N + row] = __uint_as_float(r[u]);
      } else {
#pragma unroll
        for (int u = 0; u < 32; u += 4)
          *reinterpret_cast<float4*>(ys + row * YS + 64 * half + c0 + u) =
              make_float4(__uint_as_float(r[u]), __uint_as_float(r[u + 1]),
                          __uint_as_float(r[u + 2]), __uint_as_float(r[u + 3]));
      }
    }
    if (!kT) {   // then out with consecutive threads on consecutive n, head by head
      __syncthreads();
      for (int e = tid; e < 2 * P * (N / 4); e += 256) {
        const int hh = e / (P * (N / 4)), rem = e % (P * (N / 4));
        const int pr = rem / (N / 4), c4 = 4 * (rem % (N / 4));
        float* so = states + (((int64_t)b * d.nchunks + c) * d.nheads + h0 + hh) * (int64_t)P * N;
        *reinterpret_cast<float4*>(so + (int64_t)pr * N + c4) =
            *reinterpret_cast<const float4*>(ys + pr * YS + hh * N + c4);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

// ---------------------------------------------------------------------------
// chunk_scan: one CTA per (batch x chunk, head), 256 threads; TMEM columns
// [0, 128) hold C B^T (rows i, columns j), [128, 128 + P) the output.
// Slices: N/16 of C B^T (K = dstate), N/16 of the inter-chunk term, then one
// per 16 tokens of M x (K = tokens).  kXZ: D or z given (the epilogue reads
// x and z); without them the epilogue only copies the tile out.  kS: C B^T
// is given (Sg, computed once per group by cb_tc32_kernel): no C B^T slices,
// the decay-matrix build reads it from memory, TMEM holds the output only.
// Element (i, j) of the chunk's C B^T is Sg[cf][ri][rj], (cf, ri, rj) =
// (c, i, j), or with srev (nc - 1 - c, 127 - i, 127 - j): the time-reversed
// scans of the backward, whose chunks are the forward chunks reversed.
// In a chunk of one document whose cumsum never rises (and whose 16-token
// slices decay by at most e^60 each), M's decay is split at each slice's
// last position into a row factor and a column factor carried by x, so that
// building M takes no per-element exp2 and nothing it needs is read after
// the slice's wait.
// ---------------------------------------------------------------------------
template <int P, bool kXZ, bool kS>
__global__ void __launch_bounds__(256, 2) chunk_scan_tc32_kernel(
    const float* __restrict__ x, const float* __restrict__ Bm, const float* __restrict__ Cm,
    const float* __restrict__ dtp, const float* __restrict__ cs,
    const int32_t* __restrict__ seg, const float* __restrict__ prev,
    const float* __restrict__ D, const float* __restrict__ z, Dims d, float* __restrict__ out,
    int strict, Limits lim, const float* __restrict__ Sg, int srev) {
  constexpr int PQ = P / 64;   // H row pairs / x quads per thread and slice
  constexpr int kBufK = kS ? kQ * 128 + P * 128 : kBuf;   // bytes per buffer
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = aligned_smem(smem_raw);
  __shared__ float cs_s[kQ], dt_s[kQ], sc_s[kQ], cf_s[kQ];
  __shared__ int sg_s[kQ];
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_base;
  __shared__ int ok_all;

  const int N = d.dstate;
  const int bc = blockIdx.x, h = blockIdx.y;
  const int b = bc / d.nchunks, c = bc % d.nchunks;
  const int g = h / (d.nheads / d.ngroups);
  const int64_t t0 = (int64_t)c * kQ;
  const int n = (int)min((int64_t)kQ, d.seqlen - t0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t hc = (((int64_t)b * d.nheads + h) * d.nchunks + c) * kQ;
  // the decay factors below (the decay-matrix build) need a cumsum that
  // never rises and whose 16-token slices decay by at most e^60 each
  bool mono_t = true;
  if (tid < kQ) {
    const int32_t* sp = seg ? seg + ((int64_t)b * d.nchunks + c) * kQ : nullptr;
    const float v = cs[hc + tid];
    cs_s[tid] = v;
    dt_s[tid] = dtp[hc + tid];
    sg_s[tid] = sp ? sp[tid] : 0;
    sc_s[tid] = (sp == nullptr || sp[tid] == 0) ? ex2(v * kLog2e) : 0.f;   // keep_i e^cs_i
    if (tid + 1 < kQ) mono_t = cs[hc + tid + 1] <= v;
    mono_t = mono_t && v - cs[hc + (tid | (kK - 1))] <= 60.f;
  }
  if (tid == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::mbar_fence_init();
    ok_all = 1;
  }
  constexpr uint32_t kCols = kS ? 128 : 256;
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, kCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  const bool mono = __syncthreads_and(mono_t) != 0;
  tc::fence_after_sync();
  // and a chunk of one document
  const bool factored = mono && sg_s[0] == sg_s[kQ - 1];
  // column factor of position j against the last position e of its 16-token
  // slice, e^(cs_e - cs_j) dt_j (at most dt_j); the slices' loads read it
  if (tid < kQ) cf_s[tid] = ex2((cs_s[tid | (kK - 1)] - cs_s[tid]) * kLog2e) * dt_s[tid];
  __syncthreads();
  const uint32_t tmem = tmem_base, tS = tmem, tY = kS ? tmem : tmem + 128;
  const float* Hp = prev + (((int64_t)b * d.nchunks + c) * d.nheads + h) * (int64_t)P * N;
  const float* xh = x + (int64_t)(h / d.xrep) * P;
  const float* cg = Cm + (int64_t)g * N;
  const float* bg = Bm + (int64_t)g * N;
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  // token-major operands: 4 threads per row, rows sr + 64 u, columns sk .. sk + 3
  const int sr = tid >> 2, sk = (tid & 3) * 4;
  // slices: [0, s1) C B^T, [s1, s2) inter-chunk term, [s2, nS) M x
  const int n1 = N / kK, n3 = (n + kK - 1) / kK;
  const int s1 = kS ? 0 : n1, s2 = s1 + n1, nS = s2 + n3;
  const int q = warp & 3, half = warp >> 2;
  const int i = 32 * q + lane;   // the row this thread builds M for and writes out
  const int jl = lane & 15, qh = lane >> 4;   // x^T: token in the slice, row-quad half
  // per-row values the slices reuse, read once (not on a slice's chain)
  const float cs_i = cs_s[i], sc_r0 = sc_s[sr], sc_r1 = sc_s[sr + 64];
  auto tA = [&](int u) { return base + u * kBufK; };
  auto tB = [&](int u) { return base + u * kBufK + kQ * 128; };
  // the row of the given C B^T this thread reads (kS)
  const float* srow = nullptr;
  if (kS) {
    const int cf = srev ? d.nchunks - 1 - c : c, ri = srev ? kQ - 1 - i : i;
    srow = Sg + ((((int64_t)b * d.nchunks + cf) * d.ngroups + g) * kQ + ri) * kQ;
  }

  // two register sets: slice s + 2 loads while slice s is stored / multiplied
  // (with, for a token slice, f.x = this row's factor and f.y = the column
  // factor of this lane's token, both 1 outside factored chunks)
  float4 ra0[2], rb0[2], ra1[2], rb1[2];
  float2 f0 = make_float2(1.f, 1.f), f1 = make_float2(1.f, 1.f);
  auto load_into = [&](int s, float4(&ra)[2], float4(&rb)[2], float2& f) {
    if (s < s2) {   // C (both), B (C B^T) or H (inter-chunk)
      const int k0 = kK * (s < s1 ? s : s - s1);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int r = sr + 64 * u;
        ra[u] = r < n ? ld4(cg + toff(d.sC, b, t0 + r) + k0 + sk) : zero4;
      }
      if (s < s1) {
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int r = sr + 64 * u;
          rb[u] = r < n ? ld4(bg + toff(d.sB, b, t0 + r) + k0 + sk) : zero4;
        }
      } else {
#pragma unroll
        for (int u = 0; u < PQ; ++u) rb[u] = ld4(Hp + (int64_t)(sr + 64 * u) * N + k0 + sk);
      }
    } else {            // x of tokens j0 .. j0 + 15 (16 lanes on the tokens)
      const int j0 = kK * (s - s2);
      if (factored) f = make_float2(ex2((cs_i - cs_s[j0 + kK - 1]) * kLog2e), cf_s[j0 + jl]);
      const int j = j0 + jl;
      const bool tv = j < n;
      const int64_t tx = toff(d.sx, b, t0 + (tv ? j : 0));
#pragma unroll
      for (int u = 0; u < PQ; ++u) rb[u] = tv ? ld4(xh + tx + 4 * (2 * warp + qh + 16 * u)) : zero4;
      if (kS) {         // and this row's 8 values of C B^T for the slice
        const int jb = j0 + 8 * half;
        if (32 * q + 31 < j0) {
          ra[0] = ra[1] = zero4;
        } else if (!srev) {
          ra[0] = ld4(srow + jb);
          ra[1] = ld4(srow + jb + 4);
        } else {        // columns 127 - jb - 7 .. 127 - jb, in reverse order
          const float4 lo = ld4(srow + (kQ - 8 - jb)), hi = ld4(srow + (kQ - 4 - jb));
          ra[0] = make_float4(hi.w, hi.z, hi.y, hi.x);
          ra[1] = make_float4(lo.w, lo.z, lo.y, lo.x);
        }
      }
    }
  };
  auto store_from = [&](int s, const float4(&ra)[2], const float4(&rb)[2], float2 f) {
    unsigned char* a = tA(s & 1);
    unsigned char* bt = tB(s & 1);
    if (s < s1) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        put4(a, kQ, sr + 64 * u, sk, ra[u]);
        put4(bt, kQ, sr + 64 * u, sk, rb[u]);
      }
    } else if (s < s2) {
#pragma unroll
      for (int u = 0; u < 2; ++u) put4(a, kQ, sr + 64 * u, sk, scale4(ra[u], u ? sc_r1 : sc_r0));
#pragma unroll
      for (int u = 0; u < PQ; ++u) put4(bt, P, sr + 64 * u, sk, rb[u]);
    } else {
      // M_ij = (C_i . B_j) e^(cs_i - cs_j) dt_j over j <= i (j < i if strict)
      // of one document: row i, columns j0 + 8 half .. + 7
      const int j0 = kK * (s - s2), jb = j0 + 8 * half;
      float m[8];
      if (32 * q + 31 < j0) {   // every row of this block precedes the slice
#pragma unroll
        for (int u = 0; u < 8; ++u) m[u] = 0.f;
      } else {
        uint32_t r[8];
        if (kS) {
          r[0] = __float_as_uint(ra[0].x), r[1] = __float_as_uint(ra[0].y);
          r[2] = __float_as_uint(ra[0].z), r[3] = __float_as_uint(ra[0].w);
          r[4] = __float_as_uint(ra[1].x), r[5] = __float_as_uint(ra[1].y);
          r[6] = __float_as_uint(ra[1].z), r[7] = __float_as_uint(ra[1].w);
        } else {
          asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                       : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                         "=r"(r[6]), "=r"(r[7])
                       : "r"(tS + (static_cast<uint32_t>(32 * q) << 16) + jb));
          asm volatile("tcgen05.wait::ld.sync.aligned;"
                       : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                         "+r"(r[6]), "+r"(r[7])
                       :
                       : "memory");
        }
        if (factored) {
          // e^(cs_i - cs_j) dt_j = e^(cs_i - cs_e) * e^(cs_e - cs_j) dt_j with e
          // the slice's last position: the row factor f.x here, the column
          // factor f.y on x (below); both within e^60 of 1 (rows past the
          // chunk's end are not written out)
          if (i >= j0 + kK - 1 + strict) {   // every column of the slice precedes row i
#pragma unroll
            for (int u = 0; u < 8; ++u) m[u] = __uint_as_float(r[u]) * f.x;
          } else {
#pragma unroll
            for (int u = 0; u < 8; ++u) m[u] = jb + u + strict <= i ? __uint_as_float(r[u]) * f.x : 0.f;
          }
        } else {
          const float csi = cs_s[i];
          const int sgi = sg_s[i];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int j = jb + u;
            const bool valid = j + strict <= i && j < n && sg_s[j] == sgi;
            m[u] = valid ? __uint_as_float(r[u]) * ex2((csi - cs_s[j]) * kLog2e) * dt_s[j] : 0.f;
          }
        }
      }
      put4(a, kQ, i, 8 * half, make_float4(m[0], m[1], m[2], m[3]));
      put4(a, kQ, i, 8 * half + 4, make_float4(m[4], m[5], m[6], m[7]));
      const float xs = f.y;   // token j0 + jl's column factor (1 outside factored chunks)
#pragma unroll
      for (int u = 0; u < PQ; ++u) {
        const int r = 4 * (2 * warp + qh + 16 * u);
        put1(bt, P, r, jl, rb[u].x * xs);
        put1(bt, P, r + 1, jl, rb[u].y * xs);
        put1(bt, P, r + 2, jl, rb[u].z * xs);
        put1(bt, P, r + 3, jl, rb[u].w * xs);
      }
    }
  };
  auto issue = [&](int s) {
    if (s < s1)
      mma_slice(tS, tA(s & 1), tB(s & 1), kQ, idesc_tf32(kQ, kQ), s > 0);
    else
      mma_slice(tY, tA(s & 1), tB(s & 1), P, idesc_tf32(kQ, P), s > s1);
  };

  load_into(0, ra0, rb0, f0);
  if (nS > 1) load_into(1, ra1, rb1, f1);
  bool run = true;
  for (int s = 0; run && s < nS; s += 2) {
    run = pipeline_step(s, nS, bars, tid, ok_all, lim, [&](int t) { store_from(t, ra0, rb0, f0); },
                        [&](int t) { load_into(t, ra0, rb0, f0); }, issue);
    if (run && s + 1 < nS)
      run = pipeline_step(s + 1, nS, bars, tid, ok_all, lim,
                          [&](int t) { store_from(t, ra1, rb1, f1); },
                          [&](int t) { load_into(t, ra1, rb1, f1); }, issue);
  }
  // epilogue: the output tile goes from TMEM through shared memory (rows of
  // P + 4 floats, over the tiles, which the completed MMAs no longer read),
  // then + D x and * silu(z) with consecutive threads on consecutive
  // elements of a row, rows i < n.  Each thread's elements are taken in
  // batches of 8 float4, every x / z load of a batch issued before any is
  // used; the first batch loads while the last MMAs finish.
  constexpr int kEl = kQ * (P / 4) / 256;   // float4 per thread: 8 or 16
  constexpr int kBatch = kXZ ? 8 : 1;
  float4 xv[kBatch], zv[kBatch];
  auto load_batch = [&](int bt) {
    if constexpr (kXZ) {
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = tid + 256 * (bt * kBatch + u);
        const int row = e / (P / 4), p = 4 * (e % (P / 4));
        const bool ok_row = row < n;
        xv[u] = (D && ok_row) ? ld4(x + toff(d.sx, b, t0 + row) + (int64_t)(h / d.xrep) * P + p)
                              : zero4;
        zv[u] = (z && ok_row) ? ld4(z + toff(d.sz, b, t0 + row) + (int64_t)h * P + p) : zero4;
      }
    }
  };
  if (run) load_batch(0);
  if (run) run = pipeline_drain(nS, bars, ok_all, lim);
  if (run) {
    constexpr int YS = P + 4;
    float* ys = reinterpret_cast<float*>(base);   // 128 x YS floats
#pragma unroll
    for (int c0 = 0; c0 < P / 2; c0 += 32) {
      const int col0 = half * (P / 2) + c0;
      uint32_t r[32];
      tc::tmem_ld32(tY + (static_cast<uint32_t>(32 * q) << 16) + col0, r);
      tc::tmem_ld_wait_regs(r);
#pragma unroll
      for (int u = 0; u < 32; u += 4)
        *reinterpret_cast<float4*>(ys + i * YS + col0 + u) =
            make_float4(__uint_as_float(r[u]), __uint_as_float(r[u + 1]),
                        __uint_as_float(r[u + 2]), __uint_as_float(r[u + 3]));
    }
    __syncthreads();
    const float Dh = D ? D[h] : 0.f;
#pragma unroll
    for (int bt = 0; bt < kEl / kBatch; ++bt) {
      if (bt > 0) load_batch(bt);
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int e = tid + 256 * (bt * kBatch + u);
        const int row = e / (P / 4), p = 4 * (e % (P / 4));
        if (row >= n) continue;
        float4 y = *reinterpret_cast<const float4*>(ys + row * YS + p);
        if (kXZ && D) {
          y.x = fmaf(Dh, xv[u].x, y.x);
          y.y = fmaf(Dh, xv[u].y, y.y);
          y.z = fmaf(Dh, xv[u].z, y.z);
          y.w = fmaf(Dh, xv[u].w, y.w);
        }
        if (kXZ && z) {
          y.x *= zv[u].x / (1.f + __expf(-zv[u].x));
          y.y *= zv[u].y / (1.f + __expf(-zv[u].y));
          y.z *= zv[u].z / (1.f + __expf(-zv[u].z));
          y.w *= zv[u].w / (1.f + __expf(-zv[u].w));
        }
        *reinterpret_cast<float4*>(out + (((int64_t)b * d.seqlen + t0 + row) * d.nheads + h) * P +
                                   p) = y;
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, kCols);
}


// ---------------------------------------------------------------------------
// C B^T of every (batch x chunk, group), once for all the heads of the
// group: S[b][c][g][i][j] = C_i . B_j over dstate (rows and columns past the
// sequence's end zero), and with ST its transpose.  One CTA per (batch x
// chunk, group), 256 threads, the slice pipeline above (K = dstate).
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) cb_tc32_kernel(const float* __restrict__ Bm,
                                                      const float* __restrict__ Cm, Dims d,
                                                      float* __restrict__ S,
                                                      float* __restrict__ ST, Limits lim) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* base = aligned_smem(smem_raw);
  __shared__ uint64_t bars[2];
  __shared__ uint32_t tmem_base;
  __shared__ int ok_all;
  const int N = d.dstate;
  const int bc = blockIdx.x, g = blockIdx.y;
  const int b = bc / d.nchunks, c = bc % d.nchunks;
  const int64_t t0 = (int64_t)c * kQ;
  const int n = (int)min((int64_t)kQ, d.seqlen - t0);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) {
    tc::mbar_init(&bars[0], 1);
    tc::mbar_init(&bars[1], 1);
    tc::mbar_fence_init();
    ok_all = 1;
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 128);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base;
  const float* cg = Cm + (int64_t)g * N;
  const float* bg = Bm + (int64_t)g * N;
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const int sr = tid >> 2, sk = (tid & 3) * 4;
  auto tA = [&](int u) { return base + u * kBuf; };
  auto tB = [&](int u) { return base + u * kBuf + kQ * 128; };
  const int nS = N / kK;
  float4 ra0[2], rb0[2], ra1[2], rb1[2];
  auto load_into = [&](int s, float4(&ra)[2], float4(&rb)[2]) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int r = sr + 64 * u;
      ra[u] = r < n ? ld4(cg + toff(d.sC, b, t0 + r) + kK * s + sk) : zero4;
      rb[u] = r < n ? ld4(bg + toff(d.sB, b, t0 + r) + kK * s + sk) : zero4;
    }
  };
  auto store_from = [&](int s, const float4(&ra)[2], const float4(&rb)[2]) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      put4(tA(s & 1), kQ, sr + 64 * u, sk, ra[u]);
      put4(tB(s & 1), kQ, sr + 64 * u, sk, rb[u]);
    }
  };
  auto issue = [&](int s) {
    mma_slice(tmem, tA(s & 1), tB(s & 1), kQ, idesc_tf32(kQ, kQ), s > 0);
  };
  load_into(0, ra0, rb0);
  if (nS > 1) load_into(1, ra1, rb1);
  bool run = true;
  for (int s = 0; run && s < nS; s += 2) {
    run = pipeline_step(s, nS, bars, tid, ok_all, lim, [&](int t) { store_from(t, ra0, rb0); },
                        [&](int t) { load_into(t, ra0, rb0); }, issue);
    if (run && s + 1 < nS)
      run = pipeline_step(s + 1, nS, bars, tid, ok_all, lim,
                          [&](int t) { store_from(t, ra1, rb1); },
                          [&](int t) { load_into(t, ra1, rb1); }, issue);
  }
  if (run) run = pipeline_drain(nS, bars, ok_all, lim);
  if (run) {
    const int q = warp & 3, half = warp >> 2;
    const int i = 32 * q + lane;
    const int64_t off = (((int64_t)b * d.nchunks + c) * d.ngroups + g) * kQ * kQ;
    float* srow = S + off + (int64_t)i * kQ;
#pragma unroll
    for (int c0 = 0; c0 < 64; c0 += 32) {
      const int col0 = 64 * half + c0;
      uint32_t r[32];
      tc::tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + col0, r);
      tc::tmem_ld_wait_regs(r);
#pragma unroll
      for (int u = 0; u < 32; u += 4)
        *reinterpret_cast<float4*>(srow + col0 + u) =
            make_float4(__uint_as_float(r[u]), __uint_as_float(r[u + 1]),
                        __uint_as_float(r[u + 2]), __uint_as_float(r[u + 3]));
      if (ST) {   // lanes on consecutive i: each store one 128-byte piece of a row of ST
#pragma unroll
        for (int u = 0; u < 32; ++u) ST[off + (int64_t)(col0 + u) * kQ + i] = __uint_as_float(r[u]);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 128);
}

constexpr size_t kSmem = 1024 + 2 * kBuf;   // two buffers of split tiles
// chunk_scan with C B^T given: two buffers of (128 + P) rows, or the
// epilogue's 128 x (P + 4) floats if that is more
constexpr size_t smem_scan_given(int P) {
  return 1024 + ((2 * (kQ + P) * 128 > kQ * (P + 4) * 4) ? 2 * (kQ + P) * 128
                                                           : kQ * (P + 4) * 4);
}
// chunk_scan holds 256 TMEM columns: its shared-memory request keeps it at
// two CTAs per SM, so that no third CTA waits inside tcgen05.alloc
constexpr size_t kSmemScan = 80 * 1024;

bool disabled() {
  static const bool off = [] {
    const char* e = getenv("SSD_TC32");
    return e != nullptr && e[0] == '0';
  }();
  return off;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

// Wait limit (SSD_TC32_WAIT_NS) and the test-only stall (SSD_TC32_TEST_STALL=1),
// read at every launch as the fused kernel's options are.
Limits limits() {
  Limits l{kWaitNs, 0};
  if (const char* e = getenv("SSD_TC32_WAIT_NS")) {
    const long long v = atoll(e);
    if (v > 0) l.wait_ns = (uint64_t)v;
  }
  if (const char* e = getenv("SSD_TC32_TEST_STALL")) l.stall = atoi(e) == 1;
  return l;
}
bool stride_ok(const TokStride& s) { return s.b % 4 == 0 && s.t % 4 == 0; }

template <typename K>
cudaError_t prepare(K kern, size_t bytes) {
  return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

}  // namespace tc32

bool chunk_state_tc32_fits(const float* x, const float* B, const Dims& d) {
  using namespace tc32;
  const int P = d.headdim, N = d.dstate;
  return !disabled() && d.chunk == kQ && (P == 64 || P == 128) && (N == 64 || N == 128) &&
         (P == 128 || N == 128) && aligned16(x) && aligned16(B) && stride_ok(d.sx) &&
         stride_ok(d.sB);
}

bool chunk_scan_tc32_fits(const float* x, const float* B, const float* C, const float* z,
                          const Dims& d) {
  using namespace tc32;
  const int P = d.headdim, N = d.dstate;
  return !disabled() && d.chunk == kQ && (P == 64 || P == 128) && N % 32 == 0 && N >= 32 &&
         N <= 256 && aligned16(x) && aligned16(B) && aligned16(C) && (z == nullptr || aligned16(z)) &&
         stride_ok(d.sx) && stride_ok(d.sB) && stride_ok(d.sC) && (z == nullptr || stride_ok(d.sz));
}

cudaError_t launch_chunk_state_tc32(const float* x, const float* B, const float* dtp,
                                    const float* cs, const int32_t* seg, const Dims& d,
                                    float* states, cudaStream_t st, const float* Tg) {
  using namespace tc32;
  // two heads per CTA where the per-group operand comes pre-split, the
  // per-head one has 64 rows and the two heads of a pair share the former
  const bool kT = d.dstate == 128;
  const bool pair = Tg != nullptr && d.nheads % 2 == 0 &&
                    ((kT && d.headdim == 64 && (d.nheads / d.ngroups) % 2 == 0) ||
                     (!kT && d.headdim == 128 && d.dstate == 64 && d.xrep % 2 == 0));
  if (pair) {
    dim3 g2((unsigned)(d.batch * d.nchunks), (unsigned)(d.nheads / 2));
    if (kT) {
      static cudaError_t prep = prepare(chunk_state_pair_tc32_kernel<64, 128>, kSmem);
      if (prep != cudaSuccess) return prep;
      chunk_state_pair_tc32_kernel<64, 128><<<g2, 256, kSmem, st>>>(x, B, dtp, cs, seg, d, states,
                                                                   limits(), Tg);
    } else {   // the epilogue's rows of both heads' columns need more than the two buffers
      constexpr size_t smem = 1024 + kQ * (kQ + 4) * 4;
      static cudaError_t prep = prepare(chunk_state_pair_tc32_kernel<128, 64>, smem);
      if (prep != cudaSuccess) return prep;
      chunk_state_pair_tc32_kernel<128, 64><<<g2, 256, smem, st>>>(x, B, dtp, cs, seg, d, states,
                                                                  limits(), Tg);
    }
    return cudaGetLastError();
  }
  dim3 grid((unsigned)(d.batch * d.nchunks), (unsigned)d.nheads);
#define SSD_TC32_STATE(P, N, G_)                                                                \
  if (d.headdim == P && d.dstate == N && (Tg != nullptr) == G_) {                               \
    static cudaError_t prep = prepare(chunk_state_tc32_kernel<P, N, G_>, kSmem);                \
    if (prep != cudaSuccess) return prep;                                                       \
    chunk_state_tc32_kernel<P, N, G_><<<grid, 256, kSmem, st>>>(x, B, dtp, cs, seg, d, states,  \
                                                               limits(), Tg);                   \
    return cudaGetLastError();                                                                  \
  }
  SSD_TC32_STATE(64, 128, false)
  SSD_TC32_STATE(128, 128, false)
  SSD_TC32_STATE(128, 64, false)
  SSD_TC32_STATE(64, 128, true)
  SSD_TC32_STATE(128, 128, true)
  SSD_TC32_STATE(128, 64, true)
#undef SSD_TC32_STATE
  return cudaErrorInvalidValue;
}

cudaError_t launch_group_tiles_tc32(const float* Y, TokStride sY, int groups, int64_t batch,
                                    int64_t seqlen, int nchunks, float* T, cudaStream_t st) {
  using namespace tc32;
  dim3 grid((unsigned)(batch * nchunks), (unsigned)groups, kQ / kK);
  group_tiles_kernel<<<grid, 256, 0, st>>>(Y, sY, groups, seqlen, nchunks, T);
  return cudaGetLastError();
}

bool cb_tc32_fits(const float* B, const float* C, const Dims& d) {
  using namespace tc32;
  const int N = d.dstate;
  return !disabled() && d.chunk == kQ && N % 16 == 0 && N >= 16 && N <= 256 && aligned16(B) &&
         aligned16(C) && stride_ok(d.sB) && stride_ok(d.sC);
}

cudaError_t launch_cb_tc32(const float* B, const float* C, const Dims& d, float* S, float* ST,
                           cudaStream_t st) {
  using namespace tc32;
  static cudaError_t prep = prepare(cb_tc32_kernel, kSmem);
  if (prep != cudaSuccess) return prep;
  dim3 grid((unsigned)(d.batch * d.nchunks), (unsigned)d.ngroups);
  cb_tc32_kernel<<<grid, 256, kSmem, st>>>(B, C, d, S, ST, limits());
  return cudaGetLastError();
}

cudaError_t launch_chunk_scan_tc32(const float* x, const float* B, const float* C,
                                   const float* dtp, const float* cs, const int32_t* seg,
                                   const float* prev, const float* D, const float* z,
                                   const Dims& d, float* out, cudaStream_t st, int strict,
                                   const float* Sg, int srev) {
  using namespace tc32;
  dim3 grid((unsigned)(d.batch * d.nchunks), (unsigned)d.nheads);
#define SSD_TC32_SCAN(P, XZ, S_)                                                                \
  if (d.headdim == P && (D != nullptr || z != nullptr) == XZ && (Sg != nullptr) == S_) {        \
    constexpr size_t smem = S_ ? smem_scan_given(P) : kSmemScan;                                \
    static cudaError_t prep = prepare(chunk_scan_tc32_kernel<P, XZ, S_>, smem);                 \
    if (prep != cudaSuccess) return prep;                                                       \
    chunk_scan_tc32_kernel<P, XZ, S_><<<grid, 256, smem, st>>>(                                 \
        x, B, C, dtp, cs, seg, prev, D, z, d, out, strict, limits(), Sg, srev);                 \
    return cudaGetLastError();                                                                  \
  }
  SSD_TC32_SCAN(64, true, false)
  SSD_TC32_SCAN(64, false, false)
  SSD_TC32_SCAN(128, true, false)
  SSD_TC32_SCAN(128, false, false)
  SSD_TC32_SCAN(64, true, true)
  SSD_TC32_SCAN(64, false, true)
  SSD_TC32_SCAN(128, true, true)
  SSD_TC32_SCAN(128, false, true)
#undef SSD_TC32_SCAN
  return cudaErrorInvalidValue;
}

// Status bits of the fp32 tensor-core stages' bounded waits (since the last
// reset); synchronises st.
int tc32_status(int reset, cudaStream_t st, int* bits) {
  int h = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&h, tc32::g_status32, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && reset && h != 0) {
    const int zero = 0;
    e = cudaMemcpyToSymbolAsync(tc32::g_status32, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  *bits = h;
  return static_cast<int>(e);
}

}  // namespace ssd
