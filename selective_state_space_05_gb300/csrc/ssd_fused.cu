// Fused tensor-core SSD chunk kernel for sm_103a (bf16 inputs, headdim 64,
// dstate 128, chunk 128 or 256): chunk states, inter-chunk state passing and
// chunk outputs in one persistent kernel.  Stage 1 (dt preprocessing and the
// per-chunk cumsum of dt*A) runs before it as its own kernel.
//
// Work item = (batch b, chunk c, head h), taken from an atomic ticket counter
// in chunk-major order, so an item's predecessor (b, c-1, h) always holds an
// earlier ticket.  A chunk is processed as 128-token sub-steps; per sub-step,
// with rows/columns = the sub-step's tokens and cs the chunk's cumsum:
//   CB   = C B^T                       tcgen05, A = C (K-major), B = B (K-major)
//   M    = CB o exp(cs_i - cs_j) dt_j  (j <= i, same document)   CUDA cores -> TMEM
//   Yi   = M x                         tcgen05, A = M from TMEM, B = x (MN-major)
//   Ye   = C h                         tcgen05, A = C, B = h as bf16 (MN-major)
//   H   <- exp(cs_last - cs_prev) H    CUDA cores, in TMEM (fp32 state H = h^T)
//   H   += B^T (w o x)                 tcgen05, A = B (MN-major), B = w o x (MN-major)
//          w_j = exp(cs_last - cs_j) dt_j  (the sub-step's own chunk state)
//   out  = (Yi + exp(cs_i - cs_prev) Ye + D x) * silu(z)
// where h is the state entering the sub-step; the fp32 state stays in TMEM
// (one row of dstate per TMEM lane, headdim columns) for the whole chunk.  The state entering a chunk is
// handed from item (b, c-1, h) through an L2-resident fp32 slot and a flag
// (decoupled look-back); every wait is bounded and gives up with an error
// word instead of hanging.
#include <cudaTypedefs.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace fused {

constexpr int kSub = 128;   // tokens per sub-step (MMA M)
constexpr int kP = 64;      // headdim
constexpr int kN = 128;     // dstate
constexpr int kComputeWarp0 = 2;        // warps 0 (TMA) and 1 (MMA) come first
constexpr int kSplit = 1;               // compute warps per TMEM lane quarter
constexpr int kComputeThreads = 128 * kSplit;
constexpr int kColsPerWarp = kP / kSplit;   // headdim columns each compute warp owns
constexpr int kThreads = kComputeWarp0 * 32 + kComputeThreads;
constexpr uint32_t kTmemCols = 256;
constexpr unsigned long long kWaitNs = 2000000000ull;   // any single wait: 2 s at most
constexpr uint32_t kSleepHintNs = 20000;                 // suspend hint of one try_wait

// error bits in the control block word ctrl[1]; once one is set every later
// wait of the launch returns at once, so a broken launch still ends quickly
constexpr int kErrBarrier = 1;
constexpr int kErrLookback = 2;

struct alignas(1024) Smem {
  unsigned char C[kSub * kN * 2];    // two 64-column halves, 128B swizzle
  unsigned char B[kSub * kN * 2];    // same
  unsigned char X[kSub * kP * 2];    // x; after Yi has read it: h as bf16
  unsigned char XW[kSub * kP * 2];   // w o x; after the MMAs: z, then out
  float csv[kSub];      // the sub-step's cumsum values (bulk-copied)
  float dtv[kSub];      // its dt values
  int segv[kSub];       // its reset counts
  float mcol[kSub];     // l_j - log2(dt_j): column term of the diagonal blocks
  float bcol[kSub];     // exp2(l_e - l_j) dt_j, e = last column of j's 32-block
  uint64_t full, zfull, cb, m_ready, yi_done, h_ready, y_done, tmem_free;
  uint32_t tmem_base;
  int ticket[2];
};

struct Params {
  const float* dt;       // [B, H, nc, Q]
  const float* cs;       // [B, H, nc, Q]
  const int32_t* seg;    // [B, nc, Q] or null
  const float* D;        // [H] or null
  bool has_z;
  const float* init;     // [B, H, P, N] or null
  float* final_states;   // [B, H, P, N] or null
  float* slots;          // [B*H, 2, P/4, N, 4]: hand-off states, column quads outermost
  int* flags;            // [B*H]
  int* ctrl;             // [0] ticket counter, [1] error word
  int64_t L;
  int B, H, G, Q, nc, nsub_max;
  long long items;
};

// Named barrier over a subset of warps; the non-aligned form tolerates
// threads of a warp arriving separately.
__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("barrier.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool aborted(const int* ctrl) {
  return *reinterpret_cast<const volatile int*>(ctrl + 1) != 0;
}

// Bounded wait on an mbarrier phase: gives up after kWaitNs (or at once when
// the launch has already been aborted) and records the error.
__device__ __forceinline__ void wait_or_flag(uint64_t* bar, uint32_t parity, int* ctrl) {
  if (tc::mbar_try_wait(bar, parity)) return;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (tc::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return;
    if ((i & 15u) == 0) {
      if (aborted(ctrl)) return;
      if (global_ns() - t0 > kWaitNs) {
        atomicOr(ctrl + 1, kErrBarrier);
        return;
      }
    }
  }
}

__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float tanh_fast(float v) {
  float r;
  asm("tanh.approx.f32 %0, %1;" : "=f"(r) : "f"(v));
  return r;
}
// silu(z) = z sigmoid(z) = z (1 + tanh(z/2)) / 2
__device__ __forceinline__ float silu(float v) {
  const float hv = 0.5f * v;
  return fmaf(hv, tanh_fast(hv), hv);
}

__global__ void __launch_bounds__(kThreads, 2)
    ssd_fused_kernel(const __grid_constant__ CUtensorMap map_x,
                     const __grid_constant__ CUtensorMap map_b,
                     const __grid_constant__ CUtensorMap map_c,
                     const __grid_constant__ CUtensorMap map_z,
                     const __grid_constant__ CUtensorMap map_out, Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // 1024-byte aligned start (128-byte swizzle atoms), derived from the shared
  // array itself so that accesses stay shared-memory accesses
  Smem& s = *reinterpret_cast<Smem*>(smem_raw +
                                     ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (warp == 1) {
    tc::tmem_alloc(&s.tmem_base, kTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    tc::mbar_init(&s.full, 1);
    tc::mbar_init(&s.zfull, 1);
    tc::mbar_init(&s.cb, 1);
    tc::mbar_init(&s.m_ready, 1);
    tc::mbar_init(&s.yi_done, 1);
    tc::mbar_init(&s.h_ready, 1);
    tc::mbar_init(&s.y_done, 1);
    tc::mbar_init(&s.tmem_free, 1);
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&map_x);
    tc::tma_prefetch_desc(&map_b);
    tc::tma_prefetch_desc(&map_c);
    tc::tma_prefetch_desc(&map_out);
    if (p.has_z) tc::tma_prefetch_desc(&map_z);
    s.ticket[0] = atomicAdd(p.ctrl, 1);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  const uint32_t T_A = tmem + 0;     // CB fp32 [0,128); then Yi [0,64) and Ye [64,128)
  const uint32_t T_M = tmem + 128;   // M as bf16 pairs (A operand of Yi)
  const uint32_t T_H = tmem + 192;   // fp32 state, row n = dstate index, columns = headdim

  const int pairs = p.B * p.H;
  uint32_t k = 0;   // sub-steps done by this CTA (barrier phase counter)
  for (int it = 0;; ++it) {
    __syncwarp();      // lane 0 of warp 0 wrote this ticket before reaching here
    const long long t = s.ticket[it & 1];
    __syncthreads();   // everyone has read this item's ticket
    if (t >= p.items) break;
    if (tid == 0) s.ticket[(it + 1) & 1] = atomicAdd(p.ctrl, 1);   // next item, ahead
    const int c = (int)(t / pairs);
    const int pair = (int)(t % pairs);
    const int b = pair / p.H, h = pair % p.H;
    const int g = h / (p.H / p.G);
    const int64_t t0 = (int64_t)c * p.Q;
    const int nvalid = (int)min((int64_t)p.Q, p.L - t0);
    const int nsub = (nvalid + kSub - 1) / kSub;
    const int64_t pq = ((int64_t)b * p.H + h) * p.nc + c;

    if (warp == 0) {
      // ---------------- TMA producer: a sub-step's C, B, x tiles as soon as
      // the previous sub-step's MMAs are done with them; its z tile into XW
      // once its own MMAs are done with w o x
      if (lane == 0) {
        const uint32_t vec_bytes = (p.seg ? 3u : 2u) * kSub * 4u;
        for (int sub = 0; sub < nsub; ++sub, ++k) {
          const int tok = (int)(t0 + sub * kSub);
          wait_or_flag(&s.y_done, (k & 1) ^ 1, p.ctrl);
          tc::mbar_arrive_expect_tx(&s.full, 2 * kSub * kN * 2 + kSub * kP * 2 + vec_bytes);
          tc::tma_load_4d(s.C, &map_c, &s.full, 0, g, tok, b);
          tc::tma_load_4d(s.C + kSub * 128, &map_c, &s.full, 64, g, tok, b);
          tc::tma_load_4d(s.B, &map_b, &s.full, 0, g, tok, b);
          tc::tma_load_4d(s.B + kSub * 128, &map_b, &s.full, 64, g, tok, b);
          tc::tma_load_4d(s.X, &map_x, &s.full, 0, h, tok, b);
          tc::bulk_load(s.csv, p.cs + pq * p.Q + sub * kSub, kSub * 4, &s.full);
          tc::bulk_load(s.dtv, p.dt + pq * p.Q + sub * kSub, kSub * 4, &s.full);
          if (p.seg)
            tc::bulk_load(s.segv, p.seg + ((int64_t)b * p.nc + c) * p.Q + sub * kSub, kSub * 4,
                          &s.full);
          if (p.has_z) {
            wait_or_flag(&s.y_done, k & 1, p.ctrl);
            tc::mbar_arrive_expect_tx(&s.zfull, kSub * kP * 2);
            tc::tma_load_4d(s.XW, &map_z, &s.zfull, 0, h, tok, b);
          }
        }
      } else {
        k += nsub;
      }
    } else if (warp == 1) {
      // ---------------- MMA issuer
      if (lane == 0) {
        const uint32_t sC = tc::smem_u32(s.C), sB = tc::smem_u32(s.B);
        const uint32_t sX = tc::smem_u32(s.X), sXW = tc::smem_u32(s.XW);
        constexpr uint32_t id_cb = tc::idesc_bf16(kSub, kSub, false, false);
        constexpr uint32_t id_y = tc::idesc_bf16(kSub, kP, false, true);
        constexpr uint32_t id_s = tc::idesc_bf16(kN, kP, true, true);
        for (int sub = 0; sub < nsub; ++sub, ++k) {
          const uint32_t ph = k & 1;
          wait_or_flag(&s.tmem_free, ph ^ 1, p.ctrl);
          wait_or_flag(&s.full, ph, p.ctrl);
          tc::fence_after_sync();
          for (int kk = 0; kk < 8; ++kk) {   // CB = C B^T, K = dstate
            const uint32_t ko = (kk >> 2) * (kSub * 128) + (kk & 3) * 32;
            tc::mma_ss(T_A, tc::sdesc_sw128(sC + ko, 16, 1024), tc::sdesc_sw128(sB + ko, 16, 1024),
                       id_cb, kk > 0);
          }
          tc::mma_commit(&s.cb);
          wait_or_flag(&s.m_ready, ph, p.ctrl);
          tc::fence_after_sync();
          for (int kk = 0; kk < 8; ++kk)     // Yi = M x (M holds the D skip), K = tokens
            tc::mma_ts(T_A, T_M + kk * 8, tc::sdesc_sw128(sX + kk * 2048, 16384, 1024), id_y,
                       kk > 0);
          tc::mma_commit(&s.yi_done);
          wait_or_flag(&s.h_ready, ph, p.ctrl);
          tc::fence_after_sync();
          for (int kk = 0; kk < 8; ++kk) {   // Ye = C h, K = dstate (h as bf16 in X)
            const uint32_t ko = (kk >> 2) * (kSub * 128) + (kk & 3) * 32;
            tc::mma_ss(T_A + 64, tc::sdesc_sw128(sC + ko, 16, 1024),
                       tc::sdesc_sw128(sX + kk * 2048, 16384, 1024), id_y, kk > 0);
          }
          for (int kk = 0; kk < 8; ++kk)     // H += B^T (w o x), K = tokens
            tc::mma_ss(T_H, tc::sdesc_sw128(sB + kk * 2048, kSub * 128, 1024),
                       tc::sdesc_sw128(sXW + kk * 2048, 16384, 1024), id_s, 1);
          tc::mma_commit(&s.y_done);
        }
      } else {
        k += nsub;
      }
    } else {
      // ---------------- compute: kSplit warps per TMEM lane quarter; warp
      // (quarter qr, part hc) owns row r = 32 qr + lane and its share of the
      // columns in every phase
      const int cw = warp - kComputeWarp0;
      const int qr = warp & 3;                      // TMEM lane quarter
      const int hc = cw >> 2;                       // column part, 0..kSplit-1
      const int r = qr * 32 + lane;                 // row: token (or dstate index)
      const uint32_t lane_addr = static_cast<uint32_t>(qr * 32) << 16;
      const int ct = tid - kComputeWarp0 * 32;
      const float Dh = p.D ? p.D[h] : 0.f;
      const bool has_seg = p.seg != nullptr;        // s.segv is only filled with seq_idx
      float l_prev = 0.f;
      int sg_prev = 0;

      // the state entering the chunk, this row: issued now (each thread
      // acquires the predecessor's flag itself), consumed at the first state
      // phase, so the loads overlap the first sub-step's tiles and M build
      uint32_t hin[kColsPerWarp];
      bool hin_ready = true;
      const float* hin_src = nullptr;
      if (c == 0) {
        if (p.init) {
          const float* src = p.init + ((int64_t)b * p.H + h) * kP * kN + r;
#pragma unroll
          for (int e = 0; e < kColsPerWarp; ++e)
            hin[e] = __float_as_uint(src[(hc * kColsPerWarp + e) * kN]);
        } else {
#pragma unroll
          for (int e = 0; e < kColsPerWarp; ++e) hin[e] = 0u;
        }
      } else {
        // slot layout [16 column quads][128 rows][4]: a warp's access is contiguous
        hin_src = p.slots + ((((int64_t)pair * 2 + ((c - 1) & 1)) * (kP / 4) + hc * (kColsPerWarp / 4)) *
                                 kN + r) * 4;
        int v;
        asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p.flags + pair) : "memory");
        hin_ready = v >= c;
        if (hin_ready) {
#pragma unroll
          for (int v4 = 0; v4 < kColsPerWarp / 4; ++v4)
            asm volatile("ld.relaxed.gpu.global.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(hin[4 * v4]), "=r"(hin[4 * v4 + 1]), "=r"(hin[4 * v4 + 2]),
                           "=r"(hin[4 * v4 + 3])
                         : "l"(hin_src + (int64_t)v4 * kN * 4)
                         : "memory");
        }
      }
      bool publish_pending = false;

      for (int sub = 0; sub < nsub; ++sub, ++k) {
        const uint32_t ph = k & 1;
        const int tok = sub * kSub + r;            // token within the chunk
        const bool valid = tok < nvalid;
        wait_or_flag(&s.full, ph, p.ctrl);
        // per-token scalars of the sub-step (positions past the end hold the
        // chunk's last values)
        const float l_r = s.csv[r] * kLog2e;
        const float dt_r = s.dtv[r];
        const int sg_r = has_seg ? s.segv[r] : 0;
        const float l_last = s.csv[kSub - 1] * kLog2e;
        const int sg_last = has_seg ? s.segv[kSub - 1] : 0;
        if (hc == 0) {   // one writer per row
          s.mcol[r] = dt_r > 0.f ? l_r - __log2f(dt_r) : __int_as_float(0x7f800000);
          s.bcol[r] = ex2(s.csv[r | 31] * kLog2e - l_r) * dt_r;
        }
        const float w_r = (valid && sg_r == sg_last) ? ex2(l_last - l_r) * dt_r : 0.f;
        const float rho_r = sg_r == sg_prev ? ex2(l_r - l_prev) : 0.f;
        const float carry = sg_last == sg_prev ? ex2(l_last - l_prev) : 0.f;
        named_bar_sync(1, kComputeThreads);

        // ---- M = CB o decay into T_M, 32-column blocks hc, hc + kSplit, ...
        // Below the diagonal block the decay factors as exp2(l_r - l_e) *
        // [exp2(l_e - l_j) dt_j] with e the block's last column (both <= 1);
        // the diagonal block takes one exp2 per element.  The D skip rides on
        // the diagonal: M_rr += D, so that M x includes D x_r.  Masks are selects.
        wait_or_flag(&s.cb, ph, p.ctrl);
        tc::fence_after_sync();
#pragma unroll 1
        for (int bi = 0; bi < 4 / kSplit; ++bi) {
          const int qc = hc + kSplit * bi;
          const bool live = qc <= qr;
          const bool diag = qc == qr;
          const float arow = (live && !diag) ? ex2(l_r - s.csv[qc * 32 + 31] * kLog2e) : 0.f;
#pragma unroll 1
          for (int hf = 0; hf < 2; ++hf) {
            const int c0 = qc * 32 + hf * 16;
            uint32_t packed[8];
            if (live) {
              uint32_t v[16];
              tc::tmem_ld16(T_A + lane_addr + c0, v);
              float colv[16];
              const float4* cp4 = reinterpret_cast<const float4*>((diag ? s.mcol : s.bcol) + c0);
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4) {
                const float4 f = cp4[v4];
                colv[4 * v4] = f.x;
                colv[4 * v4 + 1] = f.y;
                colv[4 * v4 + 2] = f.z;
                colv[4 * v4 + 3] = f.w;
              }
              tc::tmem_ld_wait();
              float m[16];
              if (diag) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                  const float val = __uint_as_float(v[e]) * ex2(l_r - colv[e]);
                  m[e] = (c0 + e < r) ? val : (c0 + e == r ? val + Dh : 0.f);
                }
              } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) m[e] = __uint_as_float(v[e]) * colv[e] * arow;
              }
              if (has_seg) {   // a reset between j and r zeroes the entry
                const int4* sp4 = reinterpret_cast<const int4*>(s.segv + c0);
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4) {
                  const int4 f = sp4[v4];
                  m[4 * v4] = f.x == sg_r ? m[4 * v4] : 0.f;
                  m[4 * v4 + 1] = f.y == sg_r ? m[4 * v4 + 1] : 0.f;
                  m[4 * v4 + 2] = f.z == sg_r ? m[4 * v4 + 2] : 0.f;
                  m[4 * v4 + 3] = f.w == sg_r ? m[4 * v4 + 3] : 0.f;
                }
              }
#pragma unroll
              for (int e = 0; e < 8; ++e) packed[e] = tc::pack_bf16x2(m[2 * e], m[2 * e + 1]);
            } else {
#pragma unroll
              for (int e = 0; e < 8; ++e) packed[e] = 0u;
            }
            tc::tmem_st8(T_M + lane_addr + (c0 >> 1), packed);
          }
        }
        // w o x for this warp's share of the row
        {
          const unsigned char* xr = s.X + r * 128;
          unsigned char* wr = s.XW + r * 128;
#pragma unroll
          for (int cc = 0; cc < kColsPerWarp / 8; ++cc) {
            const int ch = hc * (kColsPerWarp / 8) + cc;
            const uint32_t off = (uint32_t)((ch ^ (r & 7)) << 4);
            const uint4 xv = *reinterpret_cast<const uint4*>(xr + off);
            uint4 o;
            o.x = tc::pack_bf16x2(bf_lo(xv.x) * w_r, bf_hi(xv.x) * w_r);
            o.y = tc::pack_bf16x2(bf_lo(xv.y) * w_r, bf_hi(xv.y) * w_r);
            o.z = tc::pack_bf16x2(bf_lo(xv.z) * w_r, bf_hi(xv.z) * w_r);
            o.w = tc::pack_bf16x2(bf_lo(xv.w) * w_r, bf_hi(xv.w) * w_r);
            *reinterpret_cast<uint4*>(wr + off) = o;
          }
        }
        tc::tmem_st_wait();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        named_bar_sync(1, kComputeThreads);
        if (ct == 0) tc::mbar_arrive(&s.m_ready);

        if (sub == 0 && !hin_ready) {   // the predecessor had not handed on yet
          const unsigned long long w0 = global_ns();
          int v;
          for (uint32_t i = 0;; ++i) {
            asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p.flags + pair) : "memory");
            if (v >= c) break;
            if ((i & 63u) == 63u) {
              if (aborted(p.ctrl)) break;
              if (global_ns() - w0 > kWaitNs) {
                atomicOr(p.ctrl + 1, kErrLookback);
                break;
              }
            }
            __nanosleep(64);
          }
#pragma unroll
          for (int v4 = 0; v4 < kColsPerWarp / 4; ++v4)
            asm volatile("ld.relaxed.gpu.global.v4.b32 {%0,%1,%2,%3}, [%4];"
                         : "=r"(hin[4 * v4]), "=r"(hin[4 * v4 + 1]), "=r"(hin[4 * v4 + 2]),
                           "=r"(hin[4 * v4 + 3])
                         : "l"(hin_src + (int64_t)v4 * kN * 4)
                         : "memory");
        }

        // ---- h (entering) -> bf16 operand of Ye in X; H <- carry H in TMEM
        wait_or_flag(&s.yi_done, ph, p.ctrl);   // Yi has read x
        tc::fence_after_sync();
#pragma unroll
        for (int qd = 0; qd < kColsPerWarp / 16; ++qd) {
          const int col = hc * kColsPerWarp + qd * 16;
          uint32_t hv[16];
          if (sub == 0) {   // the entering state, from registers
#pragma unroll
            for (int e = 0; e < 16; ++e) hv[e] = hin[qd * 16 + e];
          } else {
            tc::tmem_ld16(T_H + lane_addr + col, hv);
            tc::tmem_ld_wait();
          }
          unsigned char* hr = s.X + r * 128;
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = (col >> 3) + cc;
            uint4 o;
            o.x = tc::pack_bf16x2(__uint_as_float(hv[8 * cc + 0]), __uint_as_float(hv[8 * cc + 1]));
            o.y = tc::pack_bf16x2(__uint_as_float(hv[8 * cc + 2]), __uint_as_float(hv[8 * cc + 3]));
            o.z = tc::pack_bf16x2(__uint_as_float(hv[8 * cc + 4]), __uint_as_float(hv[8 * cc + 5]));
            o.w = tc::pack_bf16x2(__uint_as_float(hv[8 * cc + 6]), __uint_as_float(hv[8 * cc + 7]));
            *reinterpret_cast<uint4*>(hr + ((ch ^ (r & 7)) << 4)) = o;
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) hv[e] = __float_as_uint(carry * __uint_as_float(hv[e]));
          tc::tmem_st16(T_H + lane_addr + col, hv);
        }
        tc::tmem_st_wait();
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        named_bar_sync(1, kComputeThreads);
        if (ct == 0) tc::mbar_arrive(&s.h_ready);

        wait_or_flag(&s.y_done, ph, p.ctrl);
        tc::fence_after_sync();

        // ---- hand the chunk's final state on (this warp's columns)
        if (sub == nsub - 1) {
          const bool last_chunk = c == p.nc - 1;
          if (!last_chunk || p.final_states) {
#pragma unroll
            for (int qd = 0; qd < kColsPerWarp / 16; ++qd) {
              const int col = hc * kColsPerWarp + qd * 16;
              uint32_t hv[16];
              tc::tmem_ld16(T_H + lane_addr + col, hv);
              tc::tmem_ld_wait();
              if (last_chunk) {
                float* dst = p.final_states + ((int64_t)b * p.H + h) * kP * kN + r;
#pragma unroll
                for (int e = 0; e < 16; ++e) dst[(col + e) * kN] = __uint_as_float(hv[e]);
              } else {
                uint4* dst = reinterpret_cast<uint4*>(p.slots) +
                             (((int64_t)pair * 2 + (c & 1)) * (kP / 4) + col / 4) * kN + r;
#pragma unroll
                for (int v4 = 0; v4 < 4; ++v4)
                  dst[v4 * kN] = make_uint4(hv[4 * v4], hv[4 * v4 + 1], hv[4 * v4 + 2], hv[4 * v4 + 3]);
              }
            }
            publish_pending = !last_chunk;   // flag raised after the epilogue
          }
        }

        // ---- epilogue: out = (Yi + rho Ye) * silu(z), z read from (and out
        // written back into) this row of XW, then one TMA store of the tile
        if (p.has_z) wait_or_flag(&s.zfull, ph, p.ctrl);
        unsigned char* zr = s.XW + r * 128;
#pragma unroll
        for (int qd = 0; qd < kColsPerWarp / 16; ++qd) {
          const int col = hc * kColsPerWarp + qd * 16;
          uint32_t yi[16], ye[16];
          tc::tmem_ld16(T_A + lane_addr + col, yi);
          tc::tmem_ld16(T_A + 64 + lane_addr + col, ye);
          tc::tmem_ld_wait();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = (col >> 3) + cc;
            uint4* slot = reinterpret_cast<uint4*>(zr + ((ch ^ (r & 7)) << 4));
            const uint4 zv = p.has_z ? *slot : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
            uint32_t o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              float y2[2];
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                const int e = cc * 8 + u * 2 + hh;
                float y = fmaf(rho_r, __uint_as_float(ye[e]), __uint_as_float(yi[e]));
                if (p.has_z) y *= silu(hh ? bf_hi(zw[u]) : bf_lo(zw[u]));
                y2[hh] = y;
              }
              o[u] = tc::pack_bf16x2(y2[0], y2[1]);
            }
            *slot = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        named_bar_sync(1, kComputeThreads);
        if (ct == 0) {
          if (publish_pending) {   // every thread's slot stores came before the barrier
            __threadfence();
            const int nv = c + 1;
            asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.flags + pair), "r"(nv)
                         : "memory");
          }
          tc::mbar_arrive(&s.tmem_free);   // Yi / Ye read out
          // rows past the sequence end are outside the tensor map and not written
          tc::tma_store_4d(&map_out, s.XW, 0, h, (int)(t0 + sub * kSub), b);
          tc::bulk_commit();
          tc::bulk_wait_read();            // XW may be rewritten after this
        }
        l_prev = l_last;
        sg_prev = sg_last;
      }
    }
  }

  // drain: the compute warps have waited for every MMA; the storing thread
  // waits for its last tile store; release TMEM
  if (tid == kComputeWarp0 * 32) tc::bulk_wait_all();
  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace fused
}  // namespace ssd

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
#include <algorithm>
#include <mutex>

namespace ssd {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// bf16 tensor [d3][d2][d1][d0] (d0 contiguous); box = 64 x 1 x 128 x 1 with the
// 128-byte swizzle, i.e. one [128 rows][64] operand block per copy; rows past
// d2 (the sequence end) are filled with zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t d3) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {d0, d1, d2, d3};
  cuuint64_t strides[3] = {d0 * 2, d0 * d1 * 2, d0 * d1 * d2 * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  if (cached[dev] == 0) {
    int n = 0;
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cached[dev] = n > 0 ? n : 148;
  }
  return cached[dev];
}

}  // namespace

bool fused_eligible(const Dims& d, bool bf16) {
  return bf16 && d.headdim == fused::kP && d.dstate == fused::kN &&
         (d.chunk == 128 || d.chunk == 256) && d.seqlen <= (int64_t)1 << 30;
}

size_t fused_ctrl_ints(const Dims& d) { return 64 + (size_t)d.batch * d.nheads; }

cudaError_t launch_fused(const __nv_bfloat16* x, const __nv_bfloat16* Bm,
                         const __nv_bfloat16* Cm, const float* dt_out, const float* cs,
                         const int32_t* seg, const float* D, const __nv_bfloat16* z,
                         const float* init, float* final_states, __nv_bfloat16* out,
                         float* slots, int* ctrl, const Dims& d, cudaStream_t st) {
  CUtensorMap mx, mb, mc, mz, mo;
  if (!make_map(&mx, x, fused::kP, d.nheads, d.seqlen, d.batch) ||
      !make_map(&mb, Bm, fused::kN, d.ngroups, d.seqlen, d.batch) ||
      !make_map(&mc, Cm, fused::kN, d.ngroups, d.seqlen, d.batch) ||
      !make_map(&mo, out, fused::kP, d.nheads, d.seqlen, d.batch))
    return cudaErrorInvalidValue;
  if (z && !make_map(&mz, z, fused::kP, d.nheads, d.seqlen, d.batch)) return cudaErrorInvalidValue;
  if (!z) mz = mx;   // never used
  cudaError_t e = cudaMemsetAsync(ctrl, 0, fused_ctrl_ints(d) * sizeof(int), st);
  if (e != cudaSuccess) return e;
  fused::Params p;
  p.dt = dt_out;
  p.cs = cs;
  p.seg = seg;
  p.D = D;
  p.has_z = z != nullptr;
  p.init = init;
  p.final_states = final_states;
  p.slots = slots;
  p.ctrl = ctrl;
  p.flags = ctrl + 64;
  p.L = d.seqlen;
  p.B = (int)d.batch;
  p.H = d.nheads;
  p.G = d.ngroups;
  p.Q = d.chunk;
  p.nc = d.nchunks;
  p.nsub_max = d.chunk / fused::kSub;
  p.items = (long long)d.batch * d.nchunks * d.nheads;
  const size_t smem = sizeof(fused::Smem) + 1024;
  static bool attr_set = false;
  if (!attr_set) {
    e = cudaFuncSetAttribute(fused::ssd_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const long long grid = std::min<long long>(p.items, 2LL * sm_count());
  fused::ssd_fused_kernel<<<(unsigned)grid, fused::kThreads, smem, st>>>(mx, mb, mc, mz, mo, p);
  return cudaGetLastError();
}

}  // namespace ssd
