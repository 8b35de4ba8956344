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
// Operands are split and written K-major into 128-byte-swizzled shared
// tiles by the CUDA cores (transposed where the token index is the K
// dimension), one 32-element K slice at a time; one thread issues the MMAs.
// The chunk_scan CTA runs three K loops: C B^T into TMEM (K = dstate), the
// inter-chunk term (e^cs C) H^T into the output accumulator (K = dstate),
// then the decay-masked matrix M = (C B^T) o L o dt, built from TMEM by the
// CUDA cores, times x (K = tokens).  Every mbarrier wait is bounded by the
// global timer and records a status bit instead of hanging.
#include <stdio.h>
#include <stdlib.h>

#include "ssd_common.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace tc32 {

__device__ int g_status32;

constexpr int kQ = 128;                       // tokens per chunk = MMA rows
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s
constexpr int kErrWait = 8;                   // status bit of a timed-out wait

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!tc::mbar_try_wait(bar, parity)) {
    if (gtimer() - t0 > kWaitNs) {
      atomicOr(&g_status32, kErrWait);
      return false;
    }
  }
  return true;
}

// byte offset of fp32 element (row, k), k < 32, in a tile of 128-byte rows
// with the 128-byte swizzle (16-byte chunks XOR row % 8)
__device__ __forceinline__ uint32_t off32(uint32_t row, uint32_t k) {
  return row * 128u + ((((k >> 2) ^ (row & 7u)) << 4) | ((k & 3u) << 2));
}

__device__ __forceinline__ void split(float v, float& hi, float& lo) {
  hi = __uint_as_float((__float_as_uint(v) + 0x1000u) & 0xFFFFE000u);   // nearest tf32
  lo = v - hi;
}

// A split tile: hi rows at t, lo rows at t + rows * 128.
__device__ __forceinline__ void put1(unsigned char* t, int rows, int r, int k, float v) {
  float hi, lo;
  split(v, hi, lo);
  const uint32_t o = off32(r, k);
  *reinterpret_cast<float*>(t + o) = hi;
  *reinterpret_cast<float*>(t + rows * 128 + o) = lo;
}
// four consecutive k (k % 4 == 0) of row r
__device__ __forceinline__ void put4(unsigned char* t, int rows, int r, int k, float4 v) {
  float4 hi, lo;
  split(v.x, hi.x, lo.x);
  split(v.y, hi.y, lo.y);
  split(v.z, hi.z, lo.z);
  split(v.w, hi.w, lo.w);
  const uint32_t o = off32(r, k);
  *reinterpret_cast<float4*>(t + o) = hi;
  *reinterpret_cast<float4*>(t + rows * 128 + o) = lo;
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

// D (+)= A B^T over one 32-wide K slice of split tiles (3 x 4 MMAs).
// a: 128 rows, b: nb rows; the first MMA overwrites D unless acc.
__device__ __forceinline__ void mma_slice(uint32_t d, const unsigned char* a,
                                          const unsigned char* b, int nb, uint32_t idesc,
                                          bool acc) {
  const uint64_t ah = tc::sdesc_sw128(tc::smem_u32(a), 16, 1024);
  const uint64_t al = tc::sdesc_sw128(tc::smem_u32(a + kQ * 128), 16, 1024);
  const uint64_t bh = tc::sdesc_sw128(tc::smem_u32(b), 16, 1024);
  const uint64_t bl = tc::sdesc_sw128(tc::smem_u32(b + nb * 128), 16, 1024);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const uint64_t o = static_cast<uint64_t>(k * 2);   // 32 bytes, in 16-byte units
    mma_tf32(d, ah + o, bh + o, idesc, (acc || k > 0) ? 1u : 0u);
    mma_tf32(d, ah + o, bl + o, idesc, 1u);
    mma_tf32(d, al + o, bh + o, idesc, 1u);
  }
}

// Makes this thread's shared stores visible to the MMAs, then syncs the CTA.
__device__ __forceinline__ void staged() {
  tc::fence_proxy_async_smem();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
}

__device__ __forceinline__ unsigned char* aligned_smem(unsigned char* raw) {
  return raw + ((1024u - (tc::smem_u32(raw) & 1023u)) & 1023u);
}

// One slice at a time: its operands are written from registers into the
// shared tiles, one thread issues its MMAs, and while they run every thread
// loads the operands of the slice after next from global memory into the
// registers just stored (two register sets, so each load has two slices'
// time to land); the tiles are written again only once the MMAs completed.

// ---------------------------------------------------------------------------
// chunk_state: one CTA per (batch x chunk, head), 256 threads.  The MMA rows
// are the 128-wide one of headdim / dstate: with dstate 128 the transposed
// state S^T = B^T (w o x) (rows n), else S = (w o x)^T B (rows p).  K = the
// chunk's tokens, 32-token slices; both operands are staged transposed
// (lane = token, rows by quads of four).
// ---------------------------------------------------------------------------
template <int P, int N>
__global__ void __launch_bounds__(256) chunk_state_tc32_kernel(
    const float* __restrict__ x, const float* __restrict__ Bm, const float* __restrict__ dtp,
    const float* __restrict__ cs, const int32_t* __restrict__ seg, Dims d,
    float* __restrict__ states) {
  constexpr bool kT = (N == 128);
  constexpr int NR = kT ? P : N;   // MMA N: the other dimension
  constexpr int XQ = P / 32, BQ = N / 32;   // float4 quads per thread and slice
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* tA = aligned_smem(smem_raw);    // 128 rows, hi + lo
  unsigned char* tB = tA + kQ * 256;             // NR rows, hi + lo
  __shared__ float wsh[kQ];
  __shared__ uint64_t bar;
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
    tc::mbar_init(&bar, 1);
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
  unsigned char* tX = kT ? tB : tA;   // (w o x)^T: P rows
  unsigned char* tBt = kT ? tA : tB;  // B^T: N rows
  constexpr uint32_t idesc = idesc_tf32(kQ, NR);
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* xh = x + (int64_t)(h / d.xrep) * P;
  const float* bg = Bm + (int64_t)g * N;

  const int ns = (n + 31) / 32;
  // two register sets: slice s + 2 loads while slice s's MMAs run
  float4 rx0[XQ], rb0[BQ], rx1[XQ], rb1[BQ];
  auto load = [&](int s, float4(&rx)[XQ], float4(&rb)[BQ]) {
    const int j = 32 * s + lane;
    const bool tv = j < n;
    const int64_t tx = toff(d.sx, b, t0 + (tv ? j : 0)), tb = toff(d.sB, b, t0 + (tv ? j : 0));
#pragma unroll
    for (int u = 0; u < XQ; ++u) rx[u] = tv ? ld4(xh + tx + 4 * (warp + 8 * u)) : zero4;
#pragma unroll
    for (int u = 0; u < BQ; ++u) rb[u] = tv ? ld4(bg + tb + 4 * (warp + 8 * u)) : zero4;
  };
  auto store = [&](int s, const float4(&rx)[XQ], const float4(&rb)[BQ]) {
    const float wj = (32 * s + lane < n) ? wsh[32 * s + lane] : 0.f;
#pragma unroll
    for (int u = 0; u < XQ; ++u) {
      const int r = 4 * (warp + 8 * u);
      put1(tX, P, r, lane, rx[u].x * wj);
      put1(tX, P, r + 1, lane, rx[u].y * wj);
      put1(tX, P, r + 2, lane, rx[u].z * wj);
      put1(tX, P, r + 3, lane, rx[u].w * wj);
    }
#pragma unroll
    for (int u = 0; u < BQ; ++u) {
      const int r = 4 * (warp + 8 * u);
      put1(tBt, N, r, lane, rb[u].x);
      put1(tBt, N, r + 1, lane, rb[u].y);
      put1(tBt, N, r + 2, lane, rb[u].z);
      put1(tBt, N, r + 3, lane, rb[u].w);
    }
  };
  // one slice: store from (rx, rb), MMAs, the load of slice s + 2 into the
  // same registers while they run, wait
  auto step = [&](int s, float4(&rx)[XQ], float4(&rb)[BQ]) -> bool {
    store(s, rx, rb);
    staged();
    if (tid == 0) {
      mma_slice(tmem, tA, tB, NR, idesc, s > 0);
      tc::mma_commit(&bar);
    }
    if (s + 2 < ns) load(s + 2, rx, rb);
    const bool ok = wait_phase(&bar, s & 1);
    if (!ok) ok_all = 0;
    tc::fence_after_sync();
    return __syncthreads_and(ok) != 0;
  };

  load(0, rx0, rb0);
  if (ns > 1) load(1, rx1, rb1);
  for (int s = 0; s < ns; s += 2) {
    if (!step(s, rx0, rb0)) break;
    if (s + 1 < ns && !step(s + 1, rx1, rb1)) break;
  }
  if (ok_all) {
    // each warp: TMEM lane quarter warp % 4, half of the NR columns
    const int q = warp & 3, half = warp >> 2;
    const int row = 32 * q + lane;   // n (kT) or p
    float* sp = states + (((int64_t)b * d.nchunks + c) * d.nheads + h) * (int64_t)P * N;
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
        float* ys = reinterpret_cast<float*>(tA);
#pragma unroll
        for (int u = 0; u < 32; u += 4)
          *reinterpret_cast<float4*>(ys + row * (N + 4) + col0 + u) =
              make_float4(__uint_as_float(r[u]), __uint_as_float(r[u + 1]),
                          __uint_as_float(r[u + 2]), __uint_as_float(r[u + 3]));
      }
    }
    if (!kT) {   // then out with consecutive threads on consecutive n
      __syncthreads();
      const float* ys = reinterpret_cast<const float*>(tA);
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
// chunk_scan: one CTA per (batch x chunk, head), 256 threads; TMEM columns
// [0, 128) hold C B^T (rows i, columns j), [128, 128 + P) the output.
// Slices: N/32 of C B^T (K = dstate), N/32 of the inter-chunk term, then one
// per 32 tokens of M x (K = tokens).
// ---------------------------------------------------------------------------
template <int P>
__global__ void __launch_bounds__(256) chunk_scan_tc32_kernel(
    const float* __restrict__ x, const float* __restrict__ Bm, const float* __restrict__ Cm,
    const float* __restrict__ dtp, const float* __restrict__ cs,
    const int32_t* __restrict__ seg, const float* __restrict__ prev,
    const float* __restrict__ D, const float* __restrict__ z, Dims d, float* __restrict__ out,
    int strict) {
  constexpr int PQ = P / 32;   // H rows / x quads per thread and slice
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* tA = aligned_smem(smem_raw);   // 128 rows, hi + lo
  unsigned char* tB = tA + kQ * 256;            // up to 128 rows, hi + lo
  __shared__ float cs_s[kQ], dt_s[kQ], sc_s[kQ];
  __shared__ int sg_s[kQ];
  __shared__ uint64_t bar;
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
  if (tid < kQ) {
    const int32_t* sp = seg ? seg + ((int64_t)b * d.nchunks + c) * kQ : nullptr;
    const float v = cs[hc + tid];
    cs_s[tid] = v;
    dt_s[tid] = dtp[hc + tid];
    sg_s[tid] = sp ? sp[tid] : 0;
    sc_s[tid] = (sp == nullptr || sp[tid] == 0) ? ex2(v * kLog2e) : 0.f;   // keep_i e^cs_i
  }
  if (tid == 0) {
    tc::mbar_init(&bar, 1);
    tc::mbar_fence_init();
    ok_all = 1;
  }
  if (warp == 0) {
    tc::tmem_alloc(&tmem_base, 256);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = tmem_base, tS = tmem, tY = tmem + 128;
  const float* Hp = prev + (((int64_t)b * d.nchunks + c) * d.nheads + h) * (int64_t)P * N;
  const float* xh = x + (int64_t)(h / d.xrep) * P;
  const float* cg = Cm + (int64_t)g * N;
  const float* bg = Bm + (int64_t)g * N;
  const float4 zero4 = make_float4(0.f, 0.f, 0.f, 0.f);
  // token-major operands: 8 threads per row, rows sr + 32 u, columns sk .. sk + 3
  const int sr = tid >> 3, sk = (tid & 7) * 4;
  const int n1 = N / 32, n3 = (n + 31) / 32, nS = 2 * n1 + n3;
  const int q = warp & 3, half = warp >> 2;
  const int i = 32 * q + lane;   // the row this thread builds M for and writes out
  // two register sets: slice s + 2 loads while slice s's MMAs run
  float4 ra0[4], rb0[4], ra1[4], rb1[4];

  auto load = [&](int s, float4(&ra)[4], float4(&rb)[4]) {
    if (s < 2 * n1) {   // C (both), B (C B^T) or H (inter-chunk)
      const int k0 = 32 * (s < n1 ? s : s - n1);
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int r = sr + 32 * u;
        ra[u] = r < n ? ld4(cg + toff(d.sC, b, t0 + r) + k0 + sk) : zero4;
      }
      if (s < n1) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = sr + 32 * u;
          rb[u] = r < n ? ld4(bg + toff(d.sB, b, t0 + r) + k0 + sk) : zero4;
        }
      } else {
#pragma unroll
        for (int u = 0; u < PQ; ++u) rb[u] = ld4(Hp + (int64_t)(sr + 32 * u) * N + k0 + sk);
      }
    } else {            // x of tokens j0 .. j0 + 31 (lane = token)
      const int j = 32 * (s - 2 * n1) + lane;
      const bool tv = j < n;
      const int64_t tx = toff(d.sx, b, t0 + (tv ? j : 0));
#pragma unroll
      for (int u = 0; u < PQ; ++u) rb[u] = tv ? ld4(xh + tx + 4 * (warp + 8 * u)) : zero4;
    }
  };
  auto store = [&](int s, const float4(&ra)[4], const float4(&rb)[4]) {
    if (s < n1) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        put4(tA, kQ, sr + 32 * u, sk, ra[u]);
        put4(tB, kQ, sr + 32 * u, sk, rb[u]);
      }
    } else if (s < 2 * n1) {
#pragma unroll
      for (int u = 0; u < 4; ++u) put4(tA, kQ, sr + 32 * u, sk, scale4(ra[u], sc_s[sr + 32 * u]));
#pragma unroll
      for (int u = 0; u < PQ; ++u) put4(tB, P, sr + 32 * u, sk, rb[u]);
    } else {
      // M_ij = (C_i . B_j) e^(cs_i - cs_j) dt_j over j <= i (j < i if strict)
      // of one document: row i, columns j0 + 16 half .. + 15
      const int j0 = 32 * (s - 2 * n1), jb = j0 + 16 * half;
      float m[16];
      if (32 * q + 31 < j0) {   // every row of this block precedes the slice
#pragma unroll
        for (int u = 0; u < 16; ++u) m[u] = 0.f;
      } else {
        uint32_t r[16];
        tc::tmem_ld16(tS + (static_cast<uint32_t>(32 * q) << 16) + jb, r);
        tc::tmem_ld_wait_regs(r);
        const float csi = cs_s[i];
        const int sgi = sg_s[i];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const int j = jb + u;
          const bool valid = j + strict <= i && j < n && sg_s[j] == sgi;
          m[u] = valid ? __uint_as_float(r[u]) * ex2((csi - cs_s[j]) * kLog2e) * dt_s[j] : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < 16; u += 4)
        put4(tA, kQ, i, 16 * half + u, make_float4(m[u], m[u + 1], m[u + 2], m[u + 3]));
#pragma unroll
      for (int u = 0; u < PQ; ++u) {
        const int r = 4 * (warp + 8 * u);
        put1(tB, P, r, lane, rb[u].x);
        put1(tB, P, r + 1, lane, rb[u].y);
        put1(tB, P, r + 2, lane, rb[u].z);
        put1(tB, P, r + 3, lane, rb[u].w);
      }
    }
  };

  auto step = [&](int s, float4(&ra)[4], float4(&rb)[4]) -> bool {
    store(s, ra, rb);
    staged();
    if (tid == 0) {
      if (s < n1)
        mma_slice(tS, tA, tB, kQ, idesc_tf32(kQ, kQ), s > 0);
      else
        mma_slice(tY, tA, tB, P, idesc_tf32(kQ, P), s > n1);
      tc::mma_commit(&bar);
    }
    if (s + 2 < nS) load(s + 2, ra, rb);
    const bool ok = wait_phase(&bar, s & 1);
    if (!ok) ok_all = 0;
    tc::fence_after_sync();
    return __syncthreads_and(ok) != 0;
  };

  load(0, ra0, rb0);
  if (nS > 1) load(1, ra1, rb1);
  for (int s = 0; s < nS; s += 2) {
    if (!step(s, ra0, rb0)) break;
    if (s + 1 < nS && !step(s + 1, ra1, rb1)) break;
  }
  // epilogue: the output tile goes from TMEM through shared memory (rows of
  // P + 4 floats, over the tiles, which the completed MMAs no longer read),
  // then + D x and * silu(z) with consecutive threads on consecutive
  // elements of a row, rows i < n
  if (ok_all) {
    constexpr int YS = P + 4;
    float* ys = reinterpret_cast<float*>(tA);   // 128 x YS floats
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
    for (int e = tid; e < n * (P / 4); e += 256) {
      const int row = e / (P / 4), p = 4 * (e % (P / 4));
      float4 y = *reinterpret_cast<const float4*>(ys + row * YS + p);
      if (D) {
        const float4 xv = ld4(x + toff(d.sx, b, t0 + row) + (int64_t)(h / d.xrep) * P + p);
        y.x = fmaf(Dh, xv.x, y.x);
        y.y = fmaf(Dh, xv.y, y.y);
        y.z = fmaf(Dh, xv.z, y.z);
        y.w = fmaf(Dh, xv.w, y.w);
      }
      if (z) {
        const float4 zv = ld4(z + toff(d.sz, b, t0 + row) + (int64_t)h * P + p);
        y.x *= zv.x / (1.f + __expf(-zv.x));
        y.y *= zv.y / (1.f + __expf(-zv.y));
        y.z *= zv.z / (1.f + __expf(-zv.z));
        y.w *= zv.w / (1.f + __expf(-zv.w));
      }
      *reinterpret_cast<float4*>(out + (((int64_t)b * d.seqlen + t0 + row) * d.nheads + h) * P +
                                 p) = y;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  if (warp == 0) tc::tmem_dealloc(tmem, 256);
}

constexpr size_t kSmem = 1024 + 2 * kQ * 256;   // two split tiles of up to 128 rows
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
                                    float* states, cudaStream_t st) {
  using namespace tc32;
  dim3 grid((unsigned)(d.batch * d.nchunks), (unsigned)d.nheads);
  cudaError_t e = cudaSuccess;
#define SSD_TC32_STATE(P, N)                                                                    \
  if (d.headdim == P && d.dstate == N) {                                                        \
    static cudaError_t prep = prepare(chunk_state_tc32_kernel<P, N>, kSmem);                          \
    if (prep != cudaSuccess) return prep;                                                       \
    chunk_state_tc32_kernel<P, N><<<grid, 256, kSmem, st>>>(x, B, dtp, cs, seg, d, states);     \
    return cudaGetLastError();                                                                  \
  }
  SSD_TC32_STATE(64, 128)
  SSD_TC32_STATE(128, 128)
  SSD_TC32_STATE(128, 64)
#undef SSD_TC32_STATE
  e = cudaErrorInvalidValue;
  return e;
}

cudaError_t launch_chunk_scan_tc32(const float* x, const float* B, const float* C,
                                   const float* dtp, const float* cs, const int32_t* seg,
                                   const float* prev, const float* D, const float* z,
                                   const Dims& d, float* out, cudaStream_t st, int strict) {
  using namespace tc32;
  dim3 grid((unsigned)(d.batch * d.nchunks), (unsigned)d.nheads);
#define SSD_TC32_SCAN(P)                                                                        \
  if (d.headdim == P) {                                                                         \
    static cudaError_t prep = prepare(chunk_scan_tc32_kernel<P>, kSmemScan);                         \
    if (prep != cudaSuccess) return prep;                                                       \
    chunk_scan_tc32_kernel<P><<<grid, 256, kSmemScan, st>>>(x, B, C, dtp, cs, seg, prev, D, z, d,    \
                                                        out, strict);                           \
    return cudaGetLastError();                                                                  \
  }
  SSD_TC32_SCAN(64)
  SSD_TC32_SCAN(128)
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
