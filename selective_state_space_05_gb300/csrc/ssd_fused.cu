// Fused tensor-core SSD kernel for sm_103a (bf16 inputs, headdim 64, dstate
// 128, chunk 128 or 256, an even number of heads per group): dt
// preprocessing and the per-chunk cumsum of dt*A, chunk states, inter-chunk
// state passing and chunk outputs in one persistent kernel, one CTA per SM.
//
// Work item = a segment of consecutive chunks (the launcher picks 1 or 2)
// of one head pair (h0 = 2 hp, h1 = h0 + 1, both in one B/C group) of one
// batch row, taken from an atomic ticket counter in segment-major order, so
// an item's predecessor (previous segment, same pair) always holds an
// earlier ticket; the state stays in TMEM across the segment's chunks.
// Warp roles:
//   warp 18   takes the tickets and, one chunk ("unit") ahead, computes the
//             per-token vectors (dt = softplus(dt_raw + dt_bias) clamped, the
//             cumsum of dt*A per head, the decay-matrix column factors, the
//             reset counts of seq_idx) into a three-slot ring
//   warp 0    lane 0 issues the TMA loads (C, B, x, z) and out stores and
//             raises the hand-off flag after a segment
//   warp 1    lane 0 issues the tcgen05 MMAs
//   warps 2-17  eight per head, one per TMEM lane quarter and headdim half
//             (four per SM sub-partition): decay matrix, state moves,
//             epilogue; they never wait for one another (every thread
//             arrives on the mbarriers its consumers wait on)
// A chunk is processed as 128-token sub-steps; per sub-step k, with rows /
// columns = the sub-step's tokens, cs the chunk's cumsum and h_e the state
// entering the sub-step (head e = 0, 1):
//   CB   = C B^T                       tcgen05, issued during step k-1's epilogue
//   M_e  = CB o exp(cs_i - cs_j) dt_j  (j <= i, same document)   CUDA cores -> TMEM
//   Yi_e = M_e x_e                     tcgen05, A = M_e from TMEM
//   H_e <- exp(cs_last - cs_prev) H_e  CUDA cores, in TMEM (fp32 state H = h^T)
//   [Ye_0 | Ye_1] = C [h_0 | h_1]      tcgen05, A = C
//   [H_0 | H_1] += B^T [w_0 o x_0 | w_1 o x_1]   one N=128 chain, A = B^T
//          w_j = exp(cs_last - cs_j) dt_j  (the sub-step's own chunk state)
//   out_e = (Yi_e + exp(cs_i - cs_prev) Ye_e + D x_e) * silu(z_e)
// Sharing the operands across the pair halves the MMA instructions per head
// (an M=128 tcgen05.mma costs about the same for N = 64 .. 256).  Only the
// state recurrence (state chain of step k -> h and carried state of step k+1)
// is serial; the rest is pipelined one step ahead: two TMEM regions trade the
// CB / Yi and M roles every step, so CB of step k+1 runs on the tensor cores
// during step k's epilogue, and x of step k+1 lands in the buffer that w o x
// of step k has left.  The compute warps convert step k+1's entering state
// while step k's Yi MMAs run.  Yi_0 and Yi_1 are committed separately so that
// each head's epilogue starts as soon as its own product is ready.  The fp32
// states stay in TMEM (one row of dstate per TMEM lane, headdim columns) for
// the whole segment and are handed to the next segment through L2-resident
// fp32 slots and a flag (decoupled look-back); every wait is bounded and
// gives up with an error word instead of hanging.
#include <cudaTypedefs.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"
#include "tc_ptx.cuh"

namespace ssd {
namespace fused {

constexpr int kSub = 128;   // tokens per sub-step (MMA M)
constexpr int kP = 64;      // headdim
constexpr int kN = 128;     // dstate
constexpr int kQmax = 256;  // largest chunk
constexpr int kRing = 3;    // units whose tickets / vectors are published
constexpr int kNH = 2;      // heads per item
constexpr int kComputeWarp0 = 2;        // warps 0 (TMA) and 1 (MMA) come first, then compute
constexpr int kHalves = 2;              // compute warps per head and TMEM lane quarter
constexpr int kPW = kP / kHalves;       // headdim columns of one compute warp
// one warp per head, headdim half and TMEM lane quarter: four per SM
// sub-partition, so that each one's latency-bound phases overlap
constexpr int kComputeThreads = 128 * kNH * kHalves;
constexpr int kVecWarp = kComputeWarp0 + kComputeThreads / 32;   // tickets and vectors
constexpr int kThreads = (kVecWarp + 1) * 32;
constexpr uint32_t kTmemCols = 512;
constexpr unsigned long long kWaitNs = 2000000000ull;   // default limit of any single wait: 2 s
constexpr uint32_t kSleepHintNs = 20000;                 // suspend hint of one try_wait

// TMEM columns: two 128-column regions R0 / R1 that trade roles every
// sub-step (CB_k then Yi_0 | Yi_1 over it in R[k%2], M_0 | M_1 in R[(k+1)%2]),
// [Ye_0 | Ye_1], [H_0 | H_1]
constexpr uint32_t kT_R0 = 0, kT_YE = 128, kT_R1 = 256, kT_H = 384;
// M_e column placement (bf16 pairs, 64 columns per head): the 16 tokens
// 16 h .. 16 h + 15 (h = 0..7, one K step of Yi_e) sit at column
// 32 (h % 2) + 8 (h / 2), so that the compute warp of headdim half hf, which
// builds the half-blocks h % 2 == hf, writes only the 32 columns of the
// region from which it read its own Yi_e half of the previous step
__host__ __device__ constexpr uint32_t m_col(int h) { return 32 * (h & 1) + 8 * (h >> 1); }

// error bits in the control block word ctrl[1] (and in the device-wide
// status word below); once one is set every later wait of the launch
// returns at once, every role stops issuing work, waits for its own copies
// and MMAs in flight, and the launch ends
constexpr int kErrBarrier = 1;
constexpr int kErrLookback = 2;
constexpr int kErrDrain = 4;   // an in-flight copy or MMA did not complete in time

// Sticky status of this device: the error bits of every launch since the
// last reset (ssd_scan_status), whatever workspace the launch used.
__device__ int g_status;

// B operand of the CB and Ye chains, K-major with the 128-byte swizzle: per
// 64-column (dstate) half, 256 rows of 128 bytes -- rows 0-127 the B tile
// (tokens), rows 128 + 64 e + p the entering state of head e, headdim p.
constexpr int kBhHalf = 256 * 128;

// One chunk of a work item: ticket t = (segment, head pair), chunk j of the
// segment.
struct Unit {
  int b, c, h0, g, pair, nvalid, nsub;   // pair = b * H/2 + h0/2
  int j, nch;                            // chunk of the segment, chunks in it
  int64_t t0;
};

struct alignas(1024) Smem {
  unsigned char C[kSub * kN * 2];      // two 64-column halves, 128B swizzle
  unsigned char BH[2 * kBhHalf];       // see kBhHalf
  // x_e of sub-step k in XB[k%2] (MN-major B operand of Yi_e); w o x_e in
  // XB[(k+1)%2] (B operand of the state chain), written over x of step k-1
  unsigned char XB[2][kNH][kSub * kP * 2];
  unsigned char Z[kNH][kSub * kP * 2];    // z_e; the epilogue writes out_e over it
  float lv[kRing][kNH][kQmax];   // l = log2(e) * cumsum of dt*A over the chunk
  float dtv[kRing][kNH][kQmax];  // dt
  float mv[kRing][kNH][kQmax];   // l_j - log2(dt_j): column term of the diagonal blocks
  float bv[kRing][kNH][kQmax];   // exp2(l_f - l_j) dt_j, f = last position of j's 32-block
  int segv[kRing][kQmax];        // reset counts (with seq_idx)
  long long tk[kRing];     // published units: ticket (>= items: no more work) ...
  Unit uk[kRing];          // ... decoded
  float dk[kRing][kNH];    // ... and the two heads' D (0 without D)
  uint64_t tk_full[kRing], tk_empty[kRing];
  uint64_t cbfull, xfull, zfull;   // C and B / x / z tiles of a sub-step landed
  uint64_t cb, yi_done[kNH], y_done;   // MMA commits: CB; Yi_e; Ye and the state chain
  uint64_t hx_ready, m_ready, out_ready;   // compute: h and w o x; M; out tile written
  uint64_t pub;            // the segment's final states are in their slots
  uint64_t mma_drain;      // every MMA the issuer started has completed (launch end)
  uint32_t tmem_base;
};

// one CTA per SM: the tiles and the alignment slack within the 227 KB a block may use
static_assert(sizeof(Smem) + 1024 <= 227 * 1024, "shared memory");

struct Params {
  // per-token vectors: computed here from the raw inputs (dt_raw != null) or
  // read from the stage-1 outputs dt / cs / seg
  const __nv_bfloat16* dt_raw;   // [B, L, H] (strides sdt_b, sdt_t, both even)
  int64_t sdt_b, sdt_t;
  const float* dt_bias;          // [H] or null
  const float* A;                // [H]
  const int32_t* seq_idx;        // [B, L] or null
  int softplus, do_clamp;
  float lo, hi;
  const float* dt;       // [B, H, nc, Q]
  const float* cs;       // [B, H, nc, Q]
  const int32_t* seg;    // [B, nc, Q] or null
  bool has_seg;          // reset counts exist (seq_idx or seg given)
  const float* D;        // [H] or null
  const __nv_bfloat16* z;   // [B, L, H, P] or null
  const float* init;     // [B, H, P, N] or null
  float* final_states;   // [B, H, P, N] or null
  float* slots;          // [B*H, 2, P/4, N, 4]: hand-off states, column quads outermost
  int* flags;            // [B * H/2]: chunks handed on per head pair
  int* ctrl;             // [0] ticket counter, [1] error word
  int64_t L;
  int B, H, G, Q, nc;
  int seg_chunks;        // chunks per work item (the state stays in TMEM across them)
  long long items;       // B * H/2 * ceil(nc / seg_chunks)
  unsigned long long wait_ns;   // limit of any single wait
  int lookback_extra;    // > 0 only in the time-out test: a hand-off flag value never reached
  int* ticket;           // the launch's work counter (ctrl[0]; ctrl[2] for the state pass)
  // state pre-pass: the state entering every segment ([B*H][nseg][P/4][N][4],
  // column quads outermost like the slots), or null: then each segment's
  // final state is handed on to the next through the slots and flags
  const float* hin;
  int nseg;
  // ... or, with hin_dense, in the chunk-state layout [B][nseg][H][P][N]
  // (stage 3's prev_states, one chunk per segment)
  bool hin_dense;
  // segment-state pass: each segment's own state, from a zero entering state
  // ([B][nseg][H][P][N]), and the decay that carries a state across the
  // segment ([B*H][nseg]; 0 when the segment holds a reset)
  float* seg_states;
  float* seg_decay;
};


__device__ __forceinline__ Unit decode(const Params& p, long long t, int j) {
  Unit u;
  const int hp = p.H / kNH;
  const int pairs = p.B * hp;
  const int sgm = (int)(t / pairs);
  u.pair = (int)(t % pairs);
  u.b = u.pair / hp;
  u.h0 = (u.pair % hp) * kNH;
  u.g = u.h0 / (p.H / p.G);
  const int c0 = sgm * p.seg_chunks;
  u.nch = min(p.seg_chunks, p.nc - c0);
  u.j = j;
  u.c = c0 + j;
  u.t0 = (int64_t)u.c * p.Q;
  u.nvalid = (int)min((int64_t)p.Q, p.L - u.t0);
  u.nsub = (u.nvalid + kSub - 1) / kSub;
  return u;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool aborted(const int* ctrl) {
  return *reinterpret_cast<const volatile int*>(ctrl + 1) != 0;
}

__device__ __forceinline__ void record_error(int* ctrl, int bits) {
  atomicOr(ctrl + 1, bits);
  atomicOr(&g_status, bits);
}

// Bounded wait on an mbarrier phase: gives up after wait_ns (or at once when
// the launch has already been aborted) and records the error.  Returns
// whether the phase completed; every caller stops issuing work after a
// failed wait.
__device__ __forceinline__ bool wait_or_flag(uint64_t* bar, uint32_t parity, int* ctrl,
                                             unsigned long long wait_ns) {
  if (tc::mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (tc::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if ((i & 15u) == 0) {
      if (aborted(ctrl)) return false;
      if (global_ns() - t0 > wait_ns) {
        record_error(ctrl, kErrBarrier);
        return false;
      }
    }
  }
}

// Wait at the end of a launch for a phase of asynchronous work this thread
// started (TMA loads, MMAs): bounded, but not cut short by an abort, so that
// nothing is still writing shared memory or TMEM when the CTA releases them.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, int* ctrl,
                                           unsigned long long wait_ns) {
  const unsigned long long t0 = global_ns();
  while (!tc::mbar_try_wait_sleep(bar, parity, kSleepHintNs)) {
    if (global_ns() - t0 > wait_ns) {
      record_error(ctrl, kErrDrain);
      return;
    }
  }
}

template <typename T>
__device__ __forceinline__ T warp_incl_scan(T v, int lane) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const T o = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v += o;
  }
  return v;
}

// The raw inputs of a unit's per-token vectors as lane `lane` of the warp
// computing them holds them: positions [lane E, lane E + E) of the chunk,
// E = Q / 32 (both heads' dt, the seq_idx values around them).  Loaded one
// unit ahead so that the loads are in flight while the warp waits.
struct VecRaw {
  float2 dt[8];
  int sq[9];   // seq_idx at positions lane E - 1 .. lane E + 7 (-1: none)
  float a[kNH], bias[kNH];   // A log2(e) and dt_bias of the two heads
  float d[kNH];              // D of the two heads (0 without D)
};

__device__ __forceinline__ void vec_load(const Params& p, const Unit& it, int lane, VecRaw& r) {
  const int E = p.Q / 32;
#pragma unroll
  for (int e = 0; e < kNH; ++e) r.d[e] = p.D ? p.D[it.h0 + e] : 0.f;
  if (p.dt_raw) {
#pragma unroll
    for (int e = 0; e < kNH; ++e) {
      r.a[e] = p.A[it.h0 + e] * kLog2e;
      r.bias[e] = p.dt_bias ? p.dt_bias[it.h0 + e] : 0.f;
    }
    // the pair's two dt values of a token are adjacent (h0 and the strides
    // are even, so each pair is one aligned 32-bit word)
    const __nv_bfloat16* src = p.dt_raw + it.b * p.sdt_b + it.t0 * p.sdt_t + it.h0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int tok = lane * E + i;
      r.dt[i] = (i < E && tok < it.nvalid)
                    ? __bfloat1622float2(
                          *reinterpret_cast<const __nv_bfloat162*>(src + (int64_t)tok * p.sdt_t))
                    : make_float2(0.f, 0.f);
    }
    if (p.seq_idx) {
      const int32_t* sq = p.seq_idx + (int64_t)it.b * p.L;
#pragma unroll
      for (int i = 0; i < 9; ++i) {
        const int tok = lane * E + i - 1;
        const int64_t gt = it.t0 + tok;
        r.sq[i] = (i <= E && tok < it.nvalid && gt >= 0) ? sq[gt] : -1;
      }
    }
  }
}

// Asynchronous 16-byte copies global -> shared (cp.async, one commit group
// per unit), so that a warp can have several units' loads in flight without
// holding them in registers.
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// The per-token vectors of both heads of one unit, written by the 32 lanes
// of a warp from what vec_load fetched.  Positions past the sequence end get
// dt = 0, so that l and the reset count keep their last values there.
// kSigned: dt may be negative (softplus off); mv then holds l itself and the
// diagonal blocks multiply by dt explicitly.  kFull: also the decay-matrix
// column factors mv and bv (the segment-state kernel needs only l, dt and
// the reset counts).
// A lane's E (4 or 8) consecutive values go to shared memory as 16-byte
// stores: E scalar stores 4 E bytes apart would conflict E ways in the banks.
__device__ __forceinline__ void store_run(int* dst, const int (&v)[8], int E) {
  int4* d4 = reinterpret_cast<int4*>(dst);
  d4[0] = make_int4(v[0], v[1], v[2], v[3]);
  if (E == 8) d4[1] = make_int4(v[4], v[5], v[6], v[7]);
}

template <bool kSigned, bool kFull = true>
__device__ __forceinline__ void vec_compute(const Params& p, const Unit& it, const VecRaw& r,
                                            float (*lv)[kQmax], float (*dtv)[kQmax],
                                            float (*mv)[kQmax], float (*bv)[kQmax], int* segv,
                                            int lane) {
  const int Q = p.Q, E = Q / 32;
  if (p.dt_raw) {
#pragma unroll
    for (int e = 0; e < kNH; ++e) {
      const float a = r.a[e], bias = r.bias[e];
      float run = 0.f, loc[8], dv[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float d = 0.f;
        if (i < E && lane * E + i < it.nvalid) {
          d = (e == 0 ? r.dt[i].x : r.dt[i].y) + bias;
          // softplus on the SFU: log(1 + exp(d)); below -15 it equals exp(d)
          // to fp32 precision, above 20 it equals d
          if (p.softplus) d = d > 20.f ? d : (d < -15.f ? __expf(d) : __logf(1.f + __expf(d)));
          if (p.do_clamp) d = fminf(fmaxf(d, p.lo), p.hi);
        }
        dv[i] = d;
        run += d * a;
        loc[i] = run;
      }
      const float excl = warp_incl_scan(run, lane) - run;
      // l at the last position of this lane's 32-block (E divides 32)
      const float lf = __shfl_sync(0xffffffffu, excl + loc[E == 8 ? 7 : 3], lane | (32 / E - 1));
#pragma unroll
      for (int h4 = 0; h4 < 8; h4 += 4) {   // four positions at a time, one 16-byte store each
        if (h4 < E) {
          float lq[4], mq[4], bq[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float l = excl + loc[h4 + i], d = dv[h4 + i];
            lq[i] = l;
            if (kFull) {
              mq[i] = kSigned ? l : (d > 0.f ? l - __log2f(d) : __int_as_float(0x7f800000));
              bq[i] = ex2(lf - l) * d;
            }
          }
          const int at = lane * E + h4;
          *reinterpret_cast<float4*>(dtv[e] + at) =
              make_float4(dv[h4], dv[h4 + 1], dv[h4 + 2], dv[h4 + 3]);
          *reinterpret_cast<float4*>(lv[e] + at) = make_float4(lq[0], lq[1], lq[2], lq[3]);
          if (kFull) {
            *reinterpret_cast<float4*>(mv[e] + at) = make_float4(mq[0], mq[1], mq[2], mq[3]);
            *reinterpret_cast<float4*>(bv[e] + at) = make_float4(bq[0], bq[1], bq[2], bq[3]);
          }
        }
      }
    }
    if (p.seq_idx) {   // a reset before token t: seq_idx[t] != seq_idx[t-1] (t >= 1)
      int cnt = 0, lc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int tok = lane * E + i;
        int f = 0;
        if (i < E && tok < it.nvalid && it.t0 + tok >= 1) f = r.sq[i + 1] != r.sq[i];
        cnt += f;
        lc[i] = cnt;
      }
      const int cex = warp_incl_scan(cnt, lane) - cnt;
#pragma unroll
      for (int i = 0; i < 8; ++i) lc[i] += cex;
      store_run(segv + lane * E, lc, E);
    }
  } else {
#pragma unroll
    for (int e = 0; e < kNH; ++e) {
      const int64_t pq = ((int64_t)it.b * p.H + it.h0 + e) * p.nc + it.c;
      for (int i = lane; i < Q; i += 32) {
        const float l = p.cs[pq * Q + i] * kLog2e, d = p.dt[pq * Q + i];
        lv[e][i] = l;
        dtv[e][i] = d;
        if (kFull) mv[e][i] = kSigned ? l : (d > 0.f ? l - __log2f(d) : __int_as_float(0x7f800000));
      }
      __syncwarp();
      if (kFull)
        for (int i = lane; i < Q; i += 32) bv[e][i] = ex2(lv[e][i | 31] - lv[e][i]) * dtv[e][i];
    }
    if (p.seg)
      for (int i = lane; i < Q; i += 32) segv[i] = p.seg[((int64_t)it.b * p.nc + it.c) * Q + i];
  }
}

// Packed pairs of fp32 (sm_100-family f32x2 arithmetic: one instruction per
// two lanes of work).
__device__ __forceinline__ uint64_t pk2(float a, float b) {
  uint64_t d;
  asm("mov.b64 %0, {%1, %2};" : "=l"(d) : "f"(a), "f"(b));
  return d;
}
__device__ __forceinline__ float2 up2(uint64_t d) {
  float2 r;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(d));
  return r;
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// the two bf16 of a 32-bit word as a packed fp32 pair (low half first)
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) {
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
// a packed fp32 pair rounded to two bf16 (low half first)
__device__ __forceinline__ uint32_t f2_to_bf2(uint64_t d) {
  const float2 f = up2(d);
  return tc::pack_bf16x2(f.x, f.y);
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

// Four column quads of one row (dstate index) of a handed-on state; quads
// are kN * 4 floats apart, so that a warp's 32 rows of one quad are contiguous.
__device__ __forceinline__ void load_slot_quads(uint32_t (&hv)[16], const float* src) {
#pragma unroll
  for (int v4 = 0; v4 < 4; ++v4)
    asm volatile("ld.relaxed.gpu.global.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(hv[4 * v4]), "=r"(hv[4 * v4 + 1]), "=r"(hv[4 * v4 + 2]), "=r"(hv[4 * v4 + 3])
                 : "l"(src + (int64_t)v4 * kN * 4)
                 : "memory");
}

template <bool kSigned>
__global__ void __launch_bounds__(kThreads, 1)
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
    tc::mbar_init(&s.cbfull, 1);
    tc::mbar_init(&s.xfull, 1);
    tc::mbar_init(&s.zfull, 1);
    tc::mbar_init(&s.cb, 1);
    for (int e = 0; e < kNH; ++e) tc::mbar_init(&s.yi_done[e], 1);
    tc::mbar_init(&s.y_done, 1);
    // arrived on by every compute thread after its own writes, so that the
    // compute warps never wait for one another
    tc::mbar_init(&s.hx_ready, kComputeThreads);
    tc::mbar_init(&s.m_ready, kComputeThreads);
    tc::mbar_init(&s.out_ready, kComputeThreads);
    tc::mbar_init(&s.pub, kComputeThreads);
    tc::mbar_init(&s.mma_drain, 1);
    for (int i = 0; i < kRing; ++i) {
      tc::mbar_init(&s.tk_full[i], 32);   // the 32 lanes of the vector warp
      tc::mbar_init(&s.tk_empty[i], 2 + kComputeThreads / 32);   // TMA, MMA lanes + compute warps
    }
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&map_x);
    tc::tma_prefetch_desc(&map_b);
    tc::tma_prefetch_desc(&map_c);
    tc::tma_prefetch_desc(&map_out);
    if (p.z) tc::tma_prefetch_desc(&map_z);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  auto W = [&](uint64_t* bar, uint32_t parity) {
    return wait_or_flag(bar, parity, p.ctrl, p.wait_ns);
  };
  // the same for all 32 lanes of a warp that then runs warp-collective code
  // (tcgen05.ld / st, shuffles): a lane stops only when the whole warp does
  auto WW = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, W(bar, parity)) != 0;
  };

  // Every role walks the same sequence of sub-steps k = 0, 1, ... (the units
  // the vector warp publishes, nsub sub-steps each); the barriers complete
  // once per sub-step, so the parity of step k is k & 1.
  if (warp == 0) {
    // ---------------- TMA: step k+1's C, B and x tiles as soon as step k's
    // Ye and state chains are done with C, B and w o x (x lands in the buffer
    // w o x of step k occupied); step k's out tiles (written over Z) once its
    // epilogue is done, then step k+1's z tiles; after a segment that hands
    // on, the flag release
    if (lane == 0) {
      int u = 0, sub = 0;
      uint32_t npub = 0;
      uint32_t n_cbx = 0, n_z = 0;   // phases armed on cbfull / xfull and on zfull
      bool live = W(&s.tk_full[0], 0);
      Unit cur = s.uk[0];
      live = live && s.tk[0] < p.items;
      tc::mbar_arrive(&s.tk_empty[0]);
      // L2: x, z and out stream through once (evict first); B and C are read
      // by every head pair of the group, the hand-off slots by the next
      // segment (both kept)
      const uint64_t pol_stream = tc::l2_policy_evict_first();
      const uint64_t pol_keep = tc::l2_policy_evict_last();
      auto load_cbx = [&](const Unit& it, int sb, int xb) {
        ++n_cbx;
        const int tok = (int)(it.t0 + sb * kSub);
        tc::mbar_arrive_expect_tx(&s.cbfull, 2 * kSub * kN * 2);
        tc::tma_load_4d_hint(s.C, &map_c, &s.cbfull, 0, it.g, tok, it.b, pol_keep);
        tc::tma_load_4d_hint(s.C + kSub * 128, &map_c, &s.cbfull, 64, it.g, tok, it.b, pol_keep);
        tc::tma_load_4d_hint(s.BH, &map_b, &s.cbfull, 0, it.g, tok, it.b, pol_keep);
        tc::tma_load_4d_hint(s.BH + kBhHalf, &map_b, &s.cbfull, 64, it.g, tok, it.b, pol_keep);
        tc::mbar_arrive_expect_tx(&s.xfull, kNH * kSub * kP * 2);
        tc::tma_load_4d_hint(s.XB[xb][0], &map_x, &s.xfull, 0, it.h0, tok, it.b, pol_stream);
        tc::tma_load_4d_hint(s.XB[xb][1], &map_x, &s.xfull, 0, it.h0 + 1, tok, it.b, pol_stream);
      };
      auto load_z = [&](const Unit& it, int sb) {
        ++n_z;
        if (p.z) {
          const int tok = (int)(it.t0 + sb * kSub);
          tc::mbar_arrive_expect_tx(&s.zfull, kNH * kSub * kP * 2);
          tc::tma_load_4d_hint(s.Z[0], &map_z, &s.zfull, 0, it.h0, tok, it.b, pol_stream);
          tc::tma_load_4d_hint(s.Z[1], &map_z, &s.zfull, 0, it.h0 + 1, tok, it.b, pol_stream);
        } else {
          tc::mbar_arrive(&s.zfull);   // Z is free for the epilogue
        }
      };
      if (live) {
        load_cbx(cur, 0, 0);
        load_z(cur, 0);
      }
      for (uint32_t k = 0; live; ++k) {
        // the step after this one: the unit's next sub-step or the next unit
        Unit nxt = cur;
        int nsb = sub + 1;
        bool has_next = true;
        if (nsb == cur.nsub) {
          const int ns = (u + 1) % kRing;
          has_next = W(&s.tk_full[ns], ((u + 1) / kRing) & 1);
          has_next = has_next && s.tk[ns] < p.items;
          nxt = s.uk[ns];
          tc::mbar_arrive(&s.tk_empty[ns]);
          nsb = 0;
        }
        // after a failed wait nothing more is issued (the launch is aborted)
        if (!W(&s.y_done, k & 1)) break;
        if (has_next) load_cbx(nxt, nsb, (k + 1) & 1);
        if (!p.hin && sub == cur.nsub - 1 && cur.j == cur.nch - 1 && cur.c < p.nc - 1) {
          // the segment's final states are in their slots once every compute
          // thread has arrived on pub; the release store orders them before
          // the flag at gpu scope (its consumer waits for flag >= its first chunk)
          if (!W(&s.pub, npub & 1)) break;
          asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p.flags + cur.pair),
                       "r"(cur.c + 1)
                       : "memory");
          ++npub;
        }
        if (!W(&s.out_ready, k & 1)) break;
        {
          // rows past the sequence end are outside the tensor map and not written
          const int tok = (int)(cur.t0 + sub * kSub);
          tc::tma_store_4d_hint(&map_out, s.Z[0], 0, cur.h0, tok, cur.b, pol_stream);
          tc::tma_store_4d_hint(&map_out, s.Z[1], 0, cur.h0 + 1, tok, cur.b, pol_stream);
          tc::bulk_commit();
        }
        if (!has_next) break;
        tc::bulk_wait_read();
        load_z(nxt, nsb);
        if (nsb == 0) ++u;
        cur = nxt;
        sub = nsb;
      }
      // the loads in flight land before the CTA may exit: every phase but the
      // last armed one of each barrier has been waited for by its consumers
      if (n_cbx > 0) {
        drain_wait(&s.cbfull, (n_cbx - 1) & 1, p.ctrl, p.wait_ns);
        drain_wait(&s.xfull, (n_cbx - 1) & 1, p.ctrl, p.wait_ns);
      }
      if (n_z > 0) drain_wait(&s.zfull, (n_z - 1) & 1, p.ctrl, p.wait_ns);
      tc::bulk_wait_all();
    }
  } else if (warp == kVecWarp) {
    // ---------------- tickets and per-token vectors: the raw inputs of the
    // next unit are loaded while the ring slot it goes to is still in use
    long long t_cur = p.items, t_pend = p.items;
    if (lane == 0) t_cur = atomicAdd(p.ticket, 1);
    t_cur = __shfl_sync(0xffffffffu, t_cur, 0);
    if (lane == 0 && t_cur < p.items) t_pend = atomicAdd(p.ticket, 1);
    int j_cur = 0;
    VecRaw raw;
    if (t_cur < p.items) vec_load(p, decode(p, t_cur, 0), lane, raw);
    for (int u = 0;; ++u) {
      const int slot = u % kRing;
      const bool ok = WW(&s.tk_empty[slot], ((u / kRing) & 1) ^ 1);
      if (t_cur < p.items)
        vec_compute<kSigned>(p, decode(p, t_cur, j_cur), raw, s.lv[slot], s.dtv[slot], s.mv[slot],
                    s.bv[slot], s.segv[slot], lane);
      if (lane == 0) {
        s.tk[slot] = t_cur;
        if (t_cur < p.items) {
          const Unit uu = decode(p, t_cur, j_cur);
          s.uk[slot] = uu;
          for (int e = 0; e < kNH; ++e) s.dk[slot][e] = raw.d[e];
        }
      }
      tc::mbar_arrive(&s.tk_full[slot]);
      if (t_cur >= p.items || !ok) break;
      if (j_cur + 1 < decode(p, t_cur, j_cur).nch) {   // the segment's next chunk
        ++j_cur;
      } else {                                          // the next item
        t_cur = __shfl_sync(0xffffffffu, t_pend, 0);
        j_cur = 0;
        if (lane == 0 && t_cur < p.items) t_pend = atomicAdd(p.ticket, 1);
      }
      if (t_cur < p.items) vec_load(p, decode(p, t_cur, j_cur), lane, raw);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer.  Per step k, in issue order:
    //   [Ye_0 | Ye_1] = C_k [h_0 | h_1]; [H_0 | H_1] += B_k^T [w o x_0 | w o x_1]
    //   Yi_e = M_e x_e (A = M_e from R[(k+1)%2], D over CB_k in R[k%2])
    //   CB_{k+1} = C_{k+1} B_{k+1}^T into R[(k+1)%2], which M_e of step k has left
    // so that CB of the next step runs during this step's epilogue.
    if (lane == 0) {
      // descriptor start addresses advance in 16-byte units: K-major k-steps
      // are 32 bytes inside a 64-column half, MN-major k-steps 8 rows of 128 bytes
      const uint64_t dC = tc::sdesc_sw128(tc::smem_u32(s.C), 16, 1024);
      const uint64_t dBH = tc::sdesc_sw128(tc::smem_u32(s.BH), 16, 1024);
      const uint64_t dBmn = tc::sdesc_sw128(tc::smem_u32(s.BH), kBhHalf, 1024);
      // x_e of buffer b starts (b kNH + e) tiles after XB (16-byte units)
      const uint64_t dX = tc::sdesc_sw128(tc::smem_u32(s.XB[0][0]), 16384, 1024);
      const uint64_t dXW = tc::sdesc_sw128(tc::smem_u32(s.XB[0][0]), kSub * kP * 2, 1024);
      constexpr uint32_t kXTile = (kSub * kP * 2) >> 4;
      auto TR = [&](uint32_t b) { return tmem + kT_R0 + b * (kT_R1 - kT_R0); };
      constexpr uint32_t id_cb = tc::idesc_bf16(kSub, 128, false, false);
      constexpr uint32_t id_y = tc::idesc_bf16(kSub, kP, false, true);
      constexpr uint32_t id_s = tc::idesc_bf16(kN, kNH * kP, true, true);
      constexpr uint32_t kHrows = (kSub * 128) >> 4;   // the h rows of [B^T | h], 16-byte units
      // CB = C B^T into TMEM columns d, K = dstate
      auto cb_chain = [&](uint32_t d) {
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t kc = ((kk >> 2) * (kSub * 128) + (kk & 3) * 32) >> 4;
          const uint32_t kb = ((kk >> 2) * kBhHalf + (kk & 3) * 32) >> 4;
          tc::mma_ss(d, dC + kc, dBH + kb, id_cb, kk > 0);
        }
      };
      int u = 0, sub = 0;
      bool live = W(&s.tk_full[0], 0);
      int nsub = s.uk[0].nsub;
      live = live && s.tk[0] < p.items;
      tc::mbar_arrive(&s.tk_empty[0]);
      if (live) {
        live = W(&s.cbfull, 0);
        tc::fence_after_sync();
        if (live) {
          cb_chain(TR(0));
          tc::mma_commit(&s.cb);
        }
      }
      // after a failed wait nothing more is issued (the launch is aborted)
      for (uint32_t k = 0; live; ++k) {
        const uint32_t ph = k & 1, bc = k & 1;
        if (!W(&s.hx_ready, ph)) break;   // h_e and w o x_e written, Ye read out
        tc::fence_after_sync();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {   // [Ye_0 | Ye_1] = C [h_0 | h_1], K = dstate
          const uint32_t kc = ((kk >> 2) * (kSub * 128) + (kk & 3) * 32) >> 4;
          const uint32_t kb = ((kk >> 2) * kBhHalf + (kk & 3) * 32) >> 4;
          tc::mma_ss(tmem + kT_YE, dC + kc, dBH + kHrows + kb, id_cb, kk > 0);
        }
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)     // [H_0 | H_1] += B^T [w o x_0 | w o x_1], K = tokens
          tc::mma_ss(tmem + kT_H, dBmn + kk * 128, dXW + (bc ^ 1) * kNH * kXTile + kk * 128, id_s, 1);
        tc::mma_commit(&s.y_done);
        if (!W(&s.m_ready, ph)) break;
        tc::fence_after_sync();
#pragma unroll
        for (int e = 0; e < kNH; ++e) {    // Yi_e = M_e x_e (M holds the D skip), K = tokens
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_ts(TR(bc) + e * kP, TR(bc ^ 1) + e * kP + m_col(kk),
                       dX + (bc * kNH + e) * kXTile + kk * 128, id_y, kk > 0);
          tc::mma_commit(&s.yi_done[e]);   // head e's epilogue may start
        }
        if (++sub == nsub) {
          ++u;
          const int ns = u % kRing;
          live = W(&s.tk_full[ns], (u / kRing) & 1);
          nsub = s.uk[ns].nsub;
          live = live && s.tk[ns] < p.items;
          tc::mbar_arrive(&s.tk_empty[ns]);
          sub = 0;
        }
        if (!live) break;
        // CB_{k+1} overwrites the columns Yi read M from: wait until Yi is done
        // (in-order execution is only promised along one accumulator)
        if (!W(&s.yi_done[kNH - 1], ph)) break;
        if (!W(&s.cbfull, ph ^ 1)) break;   // C, B of step k+1
        tc::fence_after_sync();
        cb_chain(TR(bc ^ 1));
        tc::mma_commit(&s.cb);
      }
      // every MMA issued above completes before TMEM is released
      tc::mma_commit(&s.mma_drain);
      drain_wait(&s.mma_drain, 0, p.ctrl, p.wait_ns);
    }
  } else {
    // ---------------- compute: warp (head e, half hf, quarter qr) owns row
    // r = 32 qr + lane of head e's TMEM tiles and of the sub-step's smem
    // tiles, headdim columns p0 .. p0 + 31 (and columns 16 hf .. 16 hf + 15 of
    // every 32-column block of the decay matrix).  Per
    // step k: M_e (needs CB_k) -> h and the carried state of step k+1 (needs
    // step k's state chain; the Yi MMAs run meanwhile) -> epilogue of step k
    // -> w o x_e of step k+1.  At the end of a segment the final state is
    // handed on first and the next segment's entering state is loaded after
    // the epilogue.
    const int cw = warp - kComputeWarp0;
    const int e = cw >> 3;                        // head of the pair
    const int hf = (cw >> 2) & 1;                 // half: headdim columns / decay-block columns
    const int p0 = hf * kPW;                      // first headdim column of this warp
    const int qr = warp & 3;                      // TMEM lane quarter
    const int r = qr * 32 + lane;                 // row: token (or dstate index)
    const uint32_t lane_addr = static_cast<uint32_t>(qr * 32) << 16;
    auto T_R = [&](uint32_t b) { return tmem + kT_R0 + b * (kT_R1 - kT_R0) + lane_addr; };
    const uint32_t T_YEr = tmem + kT_YE + e * kP + p0 + lane_addr;
    const uint32_t T_Hr = tmem + kT_H + e * kP + p0 + lane_addr;
    // entering-state rows of the [B^T | h] operand for this thread: dstate
    // index r is K; headdim p of head e is row 128 + 64 e + p of r's half
    unsigned char* hk = s.BH + (r >> 6) * kBhHalf + (128 + e * kP) * 128 + (r & 7) * 2;
    const int kchunk = (r & 63) >> 3;
    // h_e (entering) -> bf16 rows of the [B^T | h] operand (thread r writes
    // dstate column r of every headdim row); H_e <- carry H_e in TMEM
    auto h_convert = [&](float carry) {
      const uint64_t carry2 = pk2(carry, carry);
      tc::tmem_st_wait();   // the entering state's stores (segment start)
#pragma unroll
      for (int qd = 0; qd < kPW / 16; ++qd) {   // 16 columns at a time
        uint32_t hv[16];
        tc::tmem_ld16(T_Hr + qd * 16, hv);
        tc::tmem_ld_wait_regs(hv);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int pcol = p0 + qd * 16 + i;   // headdim p: row 128 + 64 e + p, swizzle phase p % 8
          const __nv_bfloat16 hb = __float2bfloat16_rn(__uint_as_float(hv[i]));
          *reinterpret_cast<__nv_bfloat16*>(hk + pcol * 128 + ((kchunk ^ (pcol & 7)) << 4)) = hb;
        }
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          const float2 c2 = up2(mul2(pk2(__uint_as_float(hv[i]), __uint_as_float(hv[i + 1])),
                                     carry2));
          hv[i] = __float_as_uint(c2.x);
          hv[i + 1] = __float_as_uint(c2.y);
        }
        tc::tmem_st16(T_Hr + qd * 16, hv);
      }
      tc::tmem_st_wait();
    };
    // w o x_e of a step: x from XB[xb], the product into XB[xb ^ 1]
    auto wx = [&](float w_r, int xb) {
      const unsigned char* xr = s.XB[xb][e] + r * 128;
      unsigned char* wr = s.XB[xb ^ 1][e] + r * 128;
      const uint64_t w2 = pk2(w_r, w_r);
#pragma unroll
      for (int c8 = 0; c8 < kPW / 8; ++c8) {   // 16-byte chunks of this warp's columns
        const int ch = p0 / 8 + c8;
        const uint32_t off = (uint32_t)((ch ^ (r & 7)) << 4);
        const uint4 xv = *reinterpret_cast<const uint4*>(xr + off);
        uint4 o;
        o.x = f2_to_bf2(mul2(bf2_to_f2(xv.x), w2));
        o.y = f2_to_bf2(mul2(bf2_to_f2(xv.y), w2));
        o.z = f2_to_bf2(mul2(bf2_to_f2(xv.z), w2));
        o.w = f2_to_bf2(mul2(bf2_to_f2(xv.w), w2));
        *reinterpret_cast<uint4*>(wr + off) = o;
      }
    };
    // the state entering a segment (its first chunk), this row, into T_H:
    // the initial state or zeros for chunk 0, else the predecessor segment's
    // final state once its flag is raised (it raises the flag after both
    // heads' slots are written).  Returns false when the wait for the flag
    // gave up (the launch is then aborted and nothing is stored).
    auto load_hin = [&](const Unit& it) -> bool {
      const int64_t bh = (int64_t)it.b * p.H + it.h0 + e;
      // slot layout [16 column quads][128 rows][4]: a warp's access is contiguous
      const float* slot_src =
          p.hin ? p.hin + ((bh * p.nseg + it.c / p.seg_chunks) * (kP / 4) * kN + r) * 4
                : p.slots + ((bh * 2 + ((it.c - 1) & 1)) * (kP / 4) * kN + r) * 4;
      bool ok = true;
      if (it.c > 0 && !p.hin) {
        const unsigned long long w0 = global_ns();
        int v;
        for (uint32_t i = 0;; ++i) {
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p.flags + it.pair) : "memory");
          if (v >= it.c + p.lookback_extra) break;
          if ((i & 63u) == 63u) {
            if (aborted(p.ctrl)) {
              ok = false;
              break;
            }
            if (global_ns() - w0 > p.wait_ns) {
              record_error(p.ctrl, kErrLookback);
              ok = false;
              break;
            }
          }
          __nanosleep(64);
        }
      }
      if (!__all_sync(0xffffffffu, ok)) return false;   // the whole warp stops
#pragma unroll
      for (int qd = 0; qd < kPW / 16; ++qd) {   // 16 headdim columns at a time
        const int pc = p0 + qd * 16;
        uint32_t hv[16];
        if (p.hin_dense) {   // [B][nseg][H][P][N]: row r, 16 consecutive headdim columns
          const float* src = p.hin + ((((int64_t)it.b * p.nseg + it.c / p.seg_chunks) * p.H +
                                       it.h0 + e) * kP + pc) * kN + r;
#pragma unroll
          for (int i = 0; i < 16; ++i) hv[i] = __float_as_uint(src[i * kN]);
        } else if (it.c > 0 || p.hin) {   // (the pre-pass table also holds segment 0's state)
          load_slot_quads(hv, slot_src + (int64_t)(pc / 4) * kN * 4);
        } else if (p.init) {
          const float* src = p.init + bh * kP * kN + r;
#pragma unroll
          for (int i = 0; i < 16; ++i) hv[i] = __float_as_uint(src[(pc + i) * kN]);
        } else {
#pragma unroll
          for (int i = 0; i < 16; ++i) hv[i] = 0u;
        }
        tc::tmem_st16(T_Hr + qd * 16, hv);
      }
      return true;
    };
    // per-row scalars of a step (positions past the end hold the chunk's last values)
    struct RowV {
      float l_r, l_last, dt_r;
      int sg_r, sg_last;
    };
    auto row_of = [&](int slot, int sub) {
      RowV v;
      const float* lv = s.lv[slot][e] + sub * kSub;
      const int* sgv = s.segv[slot] + sub * kSub;
      v.l_r = lv[r];
      v.l_last = lv[kSub - 1];
      v.dt_r = s.dtv[slot][e][sub * kSub + r];
      v.sg_r = p.has_seg ? sgv[r] : 0;
      v.sg_last = p.has_seg ? sgv[kSub - 1] : 0;
      return v;
    };
    // w_r = exp(cs_last - cs_r) dt_r: row r's weight in the step's own state
    auto w_of = [&](const RowV& v, int sub, int nvalid) {
      const bool valid = sub * kSub + r < nvalid;   // this row's token exists
      return (valid && v.sg_r == v.sg_last) ? ex2(v.l_last - v.l_r) * v.dt_r : 0.f;
    };

    int u = 0, slot = 0, sub = 0;
    bool live = WW(&s.tk_full[0], 0);
    live = live && s.tk[0] < p.items;
    float l_prev = 0.f;   // l and reset count where the previous sub-step of the
    int sg_prev = 0;      // chunk ended (0 at a chunk start: the cumsum restarts)
    if (live) {           // step 0: entering state, h and w o x
      const Unit& it = s.uk[0];
      live = load_hin(it);
      const RowV v = row_of(0, 0);
      if (live) h_convert(v.sg_last == 0 ? ex2(v.l_last) : 0.f);
      live = live && WW(&s.xfull, 0);
    }
    if (live) {
      const Unit& it = s.uk[0];
      const RowV v = row_of(0, 0);
      wx(w_of(v, 0, it.nvalid), 0);
      tc::fence_proxy_async_smem();   // h and w o x for the MMAs
      tc::fence_before_sync();
      tc::mbar_arrive(&s.hx_ready);
    }
    for (uint32_t k = 0; live; ++k) {
      const uint32_t ph = k & 1, bc = k & 1;
      const Unit& cur = s.uk[slot];
      const RowV v = row_of(slot, sub);
      const float l_r = v.l_r;
      const int sg_r = v.sg_r;
      const float Dh = s.dk[slot][e];
      const float* lv = s.lv[slot][e] + sub * kSub;
      const int* sgv = s.segv[slot] + sub * kSub;
      const uint32_t T_CBr = T_R(bc);              // CB_k row r
      const uint32_t T_Mr = T_R(bc ^ 1) + e * kP;  // M_e row r (bf16 pairs)

      // ---- M_e = CB o decay into TMEM, the live 32-column blocks 0..qr of
      // this row; the blocks above the diagonal are zeroed (the region held
      // Yi of step k-1).  Below the diagonal block the decay factors as
      // exp2(l_r - l_f) * [exp2(l_f - l_j) dt_j] with f the block's last
      // column (both <= 1); the diagonal block takes one exp2 per element.
      // The D skip rides on the diagonal: M_rr += D, so that M x includes
      // D x_r.  Masks are selects.
      if (!WW(&s.cb, ph)) break;
      tc::fence_after_sync();
      const float* mcol = s.mv[slot][e] + sub * kSub;
      const float* bcol = s.bv[slot][e] + sub * kSub;
#pragma unroll 1
      for (int qc = 0; qc <= qr; ++qc) {
        const bool diag = qc == qr;
        const int c0 = qc * 32 + hf * 16;   // this warp's 16 columns of the block
        uint32_t v[16];
        tc::tmem_ld16(T_CBr + c0, v);
        const float arow = diag ? 0.f : ex2(l_r - lv[qc * 32 + 31]);
        float colv[16];
        const float4* cp4 = reinterpret_cast<const float4*>((diag ? mcol : bcol) + c0);
#pragma unroll
        for (int v4 = 0; v4 < 4; ++v4) {
          const float4 f = cp4[v4];
          colv[4 * v4] = f.x;
          colv[4 * v4 + 1] = f.y;
          colv[4 * v4 + 2] = f.z;
          colv[4 * v4 + 3] = f.w;
        }
        tc::tmem_ld_wait_regs(v);
        float m[16];
        if (diag) {
          // unmasked here; D goes onto the diagonal element (column r - c0 of
          // these 16), the causal mask is applied to the packed words below
          const uint64_t lr2 = pk2(l_r, l_r), neg2 = pk2(-1.f, -1.f);
          const int t = r - c0;
          const uint64_t dpair = (t & 1) ? pk2(0.f, Dh) : pk2(Dh, 0.f);
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 d = up2(fma2(pk2(colv[i], colv[i + 1]), neg2, lr2));   // l_r - mcol
            uint64_t val = mul2(pk2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                pk2(ex2(d.x), ex2(d.y)));
            if constexpr (kSigned) {   // mcol holds l_j: the dt_j factor comes here
              const float* dcol = s.dtv[slot][e] + sub * kSub + c0;
              val = mul2(val, pk2(dcol[i], dcol[i + 1]));
            }
            if ((i >> 1) == (t >> 1)) val = add2(val, dpair);
            const float2 f = up2(val);
            m[i] = f.x;
            m[i + 1] = f.y;
          }
        } else {
          const uint64_t a2 = pk2(arow, arow);
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float2 mm = up2(mul2(pk2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])),
                                       mul2(pk2(colv[i], colv[i + 1]), a2)));
            m[i] = mm.x;
            m[i + 1] = mm.y;
          }
        }
        if (p.has_seg) {   // a reset between j and r zeroes the entry
          const int4* sp4 = reinterpret_cast<const int4*>(sgv + c0);
#pragma unroll
          for (int v4 = 0; v4 < 4; ++v4) {
            const int4 f = sp4[v4];
            m[4 * v4] = f.x == sg_r ? m[4 * v4] : 0.f;
            m[4 * v4 + 1] = f.y == sg_r ? m[4 * v4 + 1] : 0.f;
            m[4 * v4 + 2] = f.z == sg_r ? m[4 * v4 + 2] : 0.f;
            m[4 * v4 + 3] = f.w == sg_r ? m[4 * v4 + 3] : 0.f;
          }
        }
        uint32_t packed[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) packed[i] = tc::pack_bf16x2(m[2 * i], m[2 * i + 1]);
        if (diag) {
          // causal mask j <= r on the bf16 pairs: word w keeps its low half
          // when 2w <= r - c0 and its high half when 2w + 1 <= r - c0 (the
          // masked entries become exact zeros whatever their value was)
          const int s16 = 16 * (r - c0 + 1);
#pragma unroll
          for (int w = 0; w < 8; ++w)
            packed[w] &= __funnelshift_lc(0xFFFFFFFFu, 0u, (unsigned)max(s16 - 32 * w, 0));
        }
        tc::tmem_st8(T_Mr + m_col(2 * qc + hf), packed);
      }
      {
        uint32_t zero[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) zero[i] = 0u;
#pragma unroll 1
        for (int qc = qr + 1; qc < 4; ++qc) tc::tmem_st8(T_Mr + m_col(2 * qc + hf), zero);
      }
      tc::tmem_st_wait();
      tc::fence_before_sync();
      tc::mbar_arrive(&s.m_ready);

      // ---- the next step: the unit's next sub-step or the next unit's first
      int nslot = slot, nsb = sub + 1;
      bool has_next = true;
      if (nsb == cur.nsub) {
        nslot = (u + 1) % kRing;
        has_next = WW(&s.tk_full[nslot], ((u + 1) / kRing) & 1);
        has_next = has_next && s.tk[nslot] < p.items;
        nsb = 0;
      }
      const Unit& nxt = s.uk[nslot];
      const bool seg_end = sub == cur.nsub - 1 && cur.j == cur.nch - 1;
      const float lp_n = nsb == 0 ? 0.f : v.l_last;
      const int sp_n = nsb == 0 ? 0 : v.sg_last;
      RowV vn = v;
      float carry_n = 0.f;
      if (has_next) {
        vn = row_of(nslot, nsb);
        carry_n = vn.sg_last == sp_n ? ex2(vn.l_last - lp_n) : 0.f;
      }

      // ---- once step k's state chain is done: a segment's final states are
      // handed on (or written out); otherwise step k+1's h and carried state,
      // while the Yi MMAs run
      if (!WW(&s.y_done, ph)) break;
      tc::fence_after_sync();
      if (seg_end) {
        const int64_t bh = (int64_t)cur.b * p.H + cur.h0 + e;
        const bool last_chunk = cur.c == p.nc - 1;
        if (last_chunk ? p.final_states != nullptr : p.hin == nullptr) {
#pragma unroll
          for (int qd = 0; qd < kPW / 16; ++qd) {   // 16 columns at a time
            const int pc = p0 + qd * 16;
            uint32_t hv[16];
            tc::tmem_ld16(T_Hr + qd * 16, hv);
            tc::tmem_ld_wait_regs(hv);
            if (last_chunk) {
              float* dst = p.final_states + bh * kP * kN + r;
#pragma unroll
              for (int i = 0; i < 16; ++i) dst[(pc + i) * kN] = __uint_as_float(hv[i]);
            } else {
              uint4* dst = reinterpret_cast<uint4*>(p.slots) +
                           ((bh * 2 + (cur.c & 1)) * (kP / 4) + pc / 4) * kN + r;
              const uint64_t pol = tc::l2_policy_evict_last();   // read by the next segment
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst + v4 * kN),
                             "r"(hv[4 * v4]), "r"(hv[4 * v4 + 1]), "r"(hv[4 * v4 + 2]), "r"(hv[4 * v4 + 3]), "l"(pol)
                             : "memory");
            }
          }
        }
        if (!last_chunk && !p.hin) tc::mbar_arrive(&s.pub);   // warp 0 raises the flag
      } else if (has_next) {
        h_convert(carry_n);
      }

      // ---- epilogue: out_e = (Yi_e + rho Ye_e) * silu(z_e), written over
      // z_e in Z (warp 0 stores the tile); Yi_e is committed on its own, so
      // head 0 starts while Yi_1 runs
      {
        const float rho_r = sg_r == sg_prev ? ex2(l_r - l_prev) : 0.f;
        if (!WW(&s.yi_done[e], ph) || !WW(&s.zfull, ph)) break;
        tc::fence_after_sync();
        const uint32_t T_YIr = T_R(bc) + e * kP + p0;
        unsigned char* zrow = s.Z[e] + r * 128;
        const uint64_t rho2 = pk2(rho_r, rho_r), half2 = pk2(0.5f, 0.5f);
#pragma unroll
        for (int qd = 0; qd < kPW / 16; ++qd) {   // 16 columns at a time
          uint32_t yi[16], ye[16];
          tc::tmem_ld16(T_YIr + qd * 16, yi);
          tc::tmem_ld16(T_YEr + qd * 16, ye);
          tc::tmem_ld_wait_regs(yi);
          tc::tmem_ld_wait_regs(ye);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            const int ch = p0 / 8 + qd * 2 + cc;
            uint4* zp = reinterpret_cast<uint4*>(zrow + ((ch ^ (r & 7)) << 4));
            const uint4 zv = p.z ? *zp : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
            uint32_t o[4];
#pragma unroll
            for (int u4 = 0; u4 < 4; ++u4) {
              const int i = cc * 8 + u4 * 2;
              uint64_t y = fma2(rho2, pk2(__uint_as_float(ye[i]), __uint_as_float(ye[i + 1])),
                                pk2(__uint_as_float(yi[i]), __uint_as_float(yi[i + 1])));
              if (p.z) {   // silu(z) = z (1 + tanh(z/2)) / 2
                const uint64_t hz = mul2(bf2_to_f2(zw[u4]), half2);
                const float2 h = up2(hz);
                y = mul2(y, fma2(hz, pk2(tanh_fast(h.x), tanh_fast(h.y)), hz));
              }
              o[u4] = f2_to_bf2(y);
            }
            *zp = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
      }
      tc::fence_proxy_async_smem();   // out for warp 0's TMA store
      tc::fence_before_sync();
      tc::mbar_arrive(&s.out_ready);  // Yi / Ye read out, out written
      if (nsb == 0) {                 // this unit's vectors are read
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s.tk_empty[slot]);
      }
      if (!has_next) break;

      // ---- step k+1: a new segment's entering state; then w o x
      if (seg_end) {
        if (!load_hin(nxt)) break;
        h_convert(carry_n);
      }
      if (!WW(&s.xfull, ph ^ 1)) break;
      wx(w_of(vn, nsb, nxt.nvalid), bc ^ 1);
      tc::fence_proxy_async_smem();   // h and w o x for the MMAs
      tc::fence_before_sync();
      tc::mbar_arrive(&s.hx_ready);
      if (nsb == 0) {
        ++u;
        slot = nslot;
        l_prev = 0.f;
        sg_prev = 0;
      } else {
        l_prev = v.l_last;
        sg_prev = v.sg_last;
      }
      sub = nsb;
    }
  }

  // drain: the compute warps have waited for every MMA, warp 0 for its last
  // tile stores; release TMEM
  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------------------
// Segment states (the chunk-state stage at segment granularity, on tensor
// cores).  For one segment of consecutive chunks of a head pair, from a zero
// entering state:
//   S = sum_j w_j B_j (outer) x_j,  w_j = exp(cs(j -> segment end)) dt_j
// over the tokens j after the segment's last reset (w_j = 0 before it), and
// the decay that carries a state across the whole segment, exp of the sum of
// dt*A over it (0 when the segment holds a reset).  The chunks are taken
// last-first, so that the exponent of w_j, T + cs_last(chunk) - cs_j with T
// the log-decay of the chunks after j's, is known when the chunk is scaled;
// every sub-step then adds B^T [w o x_0 | w o x_1] to one TMEM accumulator
// (one N = 128 chain per sub-step, no rescaling in between).  Used by the
// state pre-pass (segments of many chunks) and, with one chunk per segment,
// as the tensor-core chunk_state stage; the per-token vectors come from
// stage 1 (dt, the per-chunk cumsum cs of dt*A, reset counts) in HBM.
// Warp roles: 0 TMA (B and x tiles, kStages deep), 1 MMA, 2-9 compute
// (head e = (warp-2)/4, token / dstate row 32 (warp%4) + lane), 10 copies
// each unit's stage-1 rows into a ring with cp.async, kSVecDepth units ahead.
// ---------------------------------------------------------------------------
constexpr int kSStages = 3;
constexpr int kSCompute = 256;
constexpr int kSVecWarp = 2 + kSCompute / 32;
constexpr int kSThreads = (kSVecWarp + 1) * 32;
constexpr uint32_t kSTmemCols = 128;
constexpr int kSRing = 6;       // published units (tickets, vectors)
constexpr int kSVecDepth = 4;   // of them, units whose copies may be in flight

struct alignas(1024) SegSmem {
  unsigned char Bt[kSStages][kSub * kN * 2];     // B tile: two 64-dstate halves, 128B swizzle
  unsigned char X[kSStages][kNH][kSub * kP * 2];  // x_e, scaled in place to w o x_e
  float csv[kSRing][kNH][kQmax];   // stage 1's cumsum of dt*A over the chunk (natural log)
  float dtv[kSRing][kNH][kQmax];   // stage 1's dt
  int segv[kSRing][kQmax];         // reset counts (with seq_idx)
  long long tk[kSRing];
  Unit uk[kSRing];
  uint64_t tk_full[kSRing], tk_empty[kSRing];
  uint64_t full[kSStages], wx[kSStages], empty[kSStages];
  uint64_t h_done, h_free, mma_drain;
  uint32_t tmem_base;
};
static_assert(sizeof(SegSmem) + 1024 <= 227 * 1024, "shared memory");

__global__ void __launch_bounds__(kSThreads, 1)
    ssd_segstate_kernel(const __grid_constant__ CUtensorMap map_x,
                        const __grid_constant__ CUtensorMap map_b, Params p) {
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  SegSmem& s = *reinterpret_cast<SegSmem*>(smem_raw +
                                           ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (warp == 1) {
    tc::tmem_alloc(&s.tmem_base, kSTmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < kSStages; ++i) {
      tc::mbar_init(&s.full[i], 1);
      tc::mbar_init(&s.wx[i], kSCompute);
      tc::mbar_init(&s.empty[i], 1);
    }
    for (int i = 0; i < kSRing; ++i) {
      tc::mbar_init(&s.tk_full[i], 32);
      tc::mbar_init(&s.tk_empty[i], 2 + kSCompute / 32);
    }
    tc::mbar_init(&s.h_done, 1);
    tc::mbar_init(&s.h_free, kSCompute);
    tc::mbar_init(&s.mma_drain, 1);
    tc::mbar_fence_init();
    tc::tma_prefetch_desc(&map_x);
    tc::tma_prefetch_desc(&map_b);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = s.tmem_base;
  auto W = [&](uint64_t* bar, uint32_t parity) {
    return wait_or_flag(bar, parity, p.ctrl, p.wait_ns);
  };
  auto WW = [&](uint64_t* bar, uint32_t parity) {
    return __all_sync(0xffffffffu, W(bar, parity)) != 0;
  };
  // Every role walks the same units (chunks, last-first within a segment) and
  // sub-steps; sub-step q of the launch uses stage q % kSStages.

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_stream = tc::l2_policy_evict_first();
      const uint64_t pol_keep = tc::l2_policy_evict_last();
      uint32_t q = 0;   // sub-steps issued
      bool ok = true;
      for (int u = 0; ok; ++u) {
        const int slot = u % kSRing;
        if (!W(&s.tk_full[slot], (u / kSRing) & 1)) break;
        const bool live = s.tk[slot] < p.items;
        const Unit it = s.uk[slot];
        tc::mbar_arrive(&s.tk_empty[slot]);
        if (!live) break;
        for (int sb = 0; sb < it.nsub; ++sb, ++q) {
          const int st = q % kSStages;
          if (q >= kSStages && !W(&s.empty[st], ((q / kSStages) - 1) & 1)) {
            ok = false;
            break;
          }
          const int tok = (int)(it.t0 + sb * kSub);
          tc::mbar_arrive_expect_tx(&s.full[st], kSub * kN * 2 + kNH * kSub * kP * 2);
          tc::tma_load_4d_hint(s.Bt[st], &map_b, &s.full[st], 0, it.g, tok, it.b, pol_keep);
          tc::tma_load_4d_hint(s.Bt[st] + kSub * 128, &map_b, &s.full[st], 64, it.g, tok, it.b,
                               pol_keep);
          tc::tma_load_4d_hint(s.X[st][0], &map_x, &s.full[st], 0, it.h0, tok, it.b, pol_stream);
          tc::tma_load_4d_hint(s.X[st][1], &map_x, &s.full[st], 0, it.h0 + 1, tok, it.b,
                               pol_stream);
        }
      }
      // the loads in flight land before the CTA may exit: the stages whose
      // last armed phase was not waited for by the MMA issuer
      for (uint32_t i = 0; i < kSStages && i < q; ++i) {
        const uint32_t last = q - 1 - i;   // one of the last kSStages sub-steps
        drain_wait(&s.full[last % kSStages], (last / kSStages) & 1, p.ctrl, p.wait_ns);
      }
    }
  } else if (warp == kSVecWarp) {
    // tickets and units (the chunks of a segment last-first), each unit's
    // stage-1 rows (cs and dt of both heads, the reset counts) copied with
    // cp.async into its ring slot; a unit is published once its copies
    // landed, kSVecDepth - 1 units behind the newest copies
    // (each unit is decoded once: decode divides 64-bit tickets)
    struct Uid {
      long long t;
      Unit it;
    };
    auto claim = [&]() {
      long long t = 0;
      if (lane == 0) t = atomicAdd(p.ticket, 1);
      return __shfl_sync(0xffffffffu, t, 0);
    };
    auto first_of = [&](long long t) {
      Uid v;
      v.t = t;
      if (t < p.items) {
        v.it = decode(p, t, 0);
        v.it = decode(p, t, v.it.nch - 1);
      }
      return v;
    };
    auto next_of = [&](const Uid& v) {
      if (v.t >= p.items) return v;
      if (v.it.j > 0) {
        Uid w = v;   // the previous chunk of the same segment
        w.it.j -= 1;
        w.it.c -= 1;
        w.it.t0 -= p.Q;
        w.it.nvalid = p.Q;   // only the sequence's last chunk can be short
        w.it.nsub = p.Q / kSub;
        return w;
      }
      return first_of(claim());
    };
    const int q4 = p.Q / 4;   // float4 / int4 per row
    // waits for the unit's ring slot, records the unit and starts its copies
    auto fill = [&](int u, const Uid& v) {
      const int slot = u % kSRing;
      const bool ok = WW(&s.tk_empty[slot], ((u / kSRing) & 1) ^ 1);
      if (lane == 0) {
        s.tk[slot] = v.t;
        if (v.t < p.items) s.uk[slot] = v.it;
      }
      if (ok && v.t < p.items) {
#pragma unroll
        for (int e = 0; e < kNH; ++e) {
          const int64_t row = (((int64_t)v.it.b * p.H + v.it.h0 + e) * p.nc + v.it.c) * p.Q;
          for (int i = lane; i < q4; i += 32) {
            cp_async16(&s.csv[slot][e][4 * i], p.cs + row + 4 * i);
            cp_async16(&s.dtv[slot][e][4 * i], p.dt + row + 4 * i);
          }
        }
        if (p.seg)
          for (int i = lane; i < q4; i += 32)
            cp_async16(&s.segv[slot][4 * i],
                       p.seg + ((int64_t)v.it.b * p.nc + v.it.c) * p.Q + 4 * i);
      }
      cp_async_commit();
      return ok;
    };
    Uid q[kSVecDepth];
    q[0] = first_of(claim());
    for (int i = 1; i < kSVecDepth; ++i) q[i] = next_of(q[i - 1]);
    bool ok = true;
    for (int i = 0; i < kSVecDepth; ++i) ok = fill(i, q[i]) && ok;
    for (int u = 0;; ++u) {
      cp_async_wait<kSVecDepth - 1>();   // unit u's copies are done (groups finish in order)
      __syncwarp();
      tc::mbar_arrive(&s.tk_full[u % kSRing]);   // each lane releases its own copies
      if (q[0].t >= p.items || !ok) break;
      const Uid nx = next_of(q[kSVecDepth - 1]);
#pragma unroll
      for (int i = 0; i < kSVecDepth - 1; ++i) q[i] = q[i + 1];
      q[kSVecDepth - 1] = nx;
      ok = fill(u + kSVecDepth, nx) && ok;
    }
    cp_async_wait<0>();   // no copy into shared memory outlives the CTA
  } else if (warp == 1) {
    if (lane == 0) {
      const uint64_t dBmn = tc::sdesc_sw128(tc::smem_u32(s.Bt[0]), kSub * 128, 1024);
      const uint64_t dXW = tc::sdesc_sw128(tc::smem_u32(s.X[0][0]), kSub * kP * 2, 1024);
      constexpr uint32_t kStageB = (kSub * kN * 2) >> 4, kStageX = (kNH * kSub * kP * 2) >> 4;
      constexpr uint32_t id_s = tc::idesc_bf16(kN, kNH * kP, true, true);
      uint32_t q = 0, items_done = 0;
      bool ok = true;
      bool first = true;   // the next MMA starts a segment (overwrites the accumulator)
      for (int u = 0; ok; ++u) {
        const int slot = u % kSRing;
        if (!W(&s.tk_full[slot], (u / kSRing) & 1)) break;
        const bool live = s.tk[slot] < p.items;
        const Unit it = s.uk[slot];
        tc::mbar_arrive(&s.tk_empty[slot]);
        if (!live) break;
        if (first && items_done > 0 && !W(&s.h_free, (items_done - 1) & 1)) break;
        for (int sb = 0; sb < it.nsub; ++sb, ++q) {
          const int st = q % kSStages;
          if (!W(&s.wx[st], (q / kSStages) & 1)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc::mma_ss(tmem, dBmn + st * kStageB + kk * 128, dXW + st * kStageX + kk * 128, id_s,
                       first ? (kk > 0) : 1);
          first = false;
          tc::mma_commit(&s.empty[st]);   // the stage may be reloaded
        }
        if (ok && it.j == 0) {   // the segment's first chunk comes last
          tc::mma_commit(&s.h_done);
          ++items_done;
          first = true;
        }
      }
      tc::mma_commit(&s.mma_drain);
      drain_wait(&s.mma_drain, 0, p.ctrl, p.wait_ns);
    }
  } else {
    // compute: scale x rows by w in place; at a segment's end read the state
    const int cw = warp - 2;
    const int e = cw >> 2;
    const int qr = warp & 3;
    const int r = qr * 32 + lane;
    const uint32_t lane_addr = static_cast<uint32_t>(qr * 32) << 16;
    uint32_t q = 0, items_done = 0;
    float T = 0.f;          // log2-decay of the segment's chunks after the current one
    bool reset_later = false;
    for (int u = 0;; ++u) {
      const int slot = u % kSRing;
      if (!WW(&s.tk_full[slot], (u / kSRing) & 1)) break;
      const bool live = s.tk[slot] < p.items;
      const Unit it = s.uk[slot];
      if (!live) {
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&s.tk_empty[slot]);
        break;
      }
      if (it.j == it.nch - 1) {   // a segment starts (its last chunk comes first)
        T = 0.f;
        reset_later = false;
      }
      const float* lv = s.csv[slot][e];   // natural log: times log2(e) below
      const float l_last = lv[p.Q - 1] * kLog2e;
      const int sg_last = p.has_seg ? s.segv[slot][p.Q - 1] : 0;
      bool ok = true;
      for (int sb = 0; sb < it.nsub; ++sb, ++q) {
        const int st = q % kSStages;
        const int tok = sb * kSub + r;
        float w = 0.f;
        if (tok < it.nvalid && !reset_later && (!p.has_seg || s.segv[slot][tok] == sg_last))
          w = ex2(fmaf(-lv[tok], kLog2e, T + l_last)) * s.dtv[slot][e][tok];
        if (!WW(&s.full[st], (q / kSStages) & 1)) {
          ok = false;
          break;
        }
        unsigned char* xr = s.X[st][e] + r * 128;
        const uint64_t w2 = pk2(w, w);
#pragma unroll
        for (int c8 = 0; c8 < 8; ++c8) {
          // the row's 64 columns, in place, in the tile's swizzled chunk
          // order: the 8 rows of a phase then hit 8 different bank groups
          uint4* ptr = reinterpret_cast<uint4*>(xr + ((c8 ^ (r & 7)) << 4));
          const uint4 xv = *ptr;
          uint4 o;
          o.x = f2_to_bf2(mul2(bf2_to_f2(xv.x), w2));
          o.y = f2_to_bf2(mul2(bf2_to_f2(xv.y), w2));
          o.z = f2_to_bf2(mul2(bf2_to_f2(xv.z), w2));
          o.w = f2_to_bf2(mul2(bf2_to_f2(xv.w), w2));
          *ptr = o;
        }
        tc::fence_proxy_async_smem();
        tc::mbar_arrive(&s.wx[st]);
      }
      T += l_last;
      reset_later = reset_later || sg_last > 0;
      __syncwarp();
      if (lane == 0) tc::mbar_arrive(&s.tk_empty[slot]);
      if (!ok) break;
      if (it.j == 0) {   // the segment is complete: S and its decay
        if (!WW(&s.h_done, items_done & 1)) break;
        tc::fence_after_sync();
        const int sgm = it.c / p.seg_chunks;
        const int h = it.h0 + e;
        float* dst = p.seg_states +
                     ((((int64_t)it.b * p.nseg + sgm) * p.H + h) * kP) * kN + r;
#pragma unroll
        for (int qd = 0; qd < kP / 16; ++qd) {
          uint32_t hv[16];
          tc::tmem_ld16(tmem + e * kP + qd * 16 + lane_addr, hv);
          tc::tmem_ld_wait_regs(hv);
#pragma unroll
          for (int i = 0; i < 16; ++i) dst[(qd * 16 + i) * kN] = __uint_as_float(hv[i]);
        }
        if (r == 0 && p.seg_decay)
          p.seg_decay[((int64_t)it.b * p.H + h) * p.nseg + sgm] = reset_later ? 0.f : ex2(T);
        tc::fence_before_sync();
        tc::mbar_arrive(&s.h_free);
        ++items_done;
      }
    }
  }
  __syncwarp();
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 1) tc::tmem_dealloc(tmem, kSTmemCols);
}

// The state entering every segment: h_0 = initial state (or 0),
// h_{s+1} = decay_s h_s + S_s, written in the slot layout ([P/4][N][4] per
// (b h, segment)) that the fused kernel reads.  One thread per (b h, column
// quad, dstate row).
__global__ void __launch_bounds__(256)
    segment_passing_kernel(const float* __restrict__ seg_states,
                           const float* __restrict__ seg_decay, const float* __restrict__ init,
                           float* __restrict__ hin, int B, int H, int nseg) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t per_bh = (kP / 4) * kN;
  if (idx >= (int64_t)B * H * per_bh) return;
  const int64_t bh = idx / per_bh;
  const int quad = (int)((idx % per_bh) / kN), n = (int)(idx % kN);
  const int b = (int)(bh / H), h = (int)(bh % H);
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (init) {
    const float* src = init + bh * kP * kN + (quad * 4) * kN + n;
    v = make_float4(src[0], src[kN], src[2 * kN], src[3 * kN]);
  }
  for (int sg = 0; sg < nseg; ++sg) {
    reinterpret_cast<float4*>(hin)[(bh * nseg + sg) * per_bh + quad * kN + n] = v;
    const float dcy = seg_decay[bh * nseg + sg];
    const float* S = seg_states + (((int64_t)b * nseg + sg) * H + h) * kP * kN +
                     (quad * 4) * kN + n;
    v.x = fmaf(dcy, v.x, S[0]);
    v.y = fmaf(dcy, v.y, S[kN]);
    v.z = fmaf(dcy, v.z, S[2 * kN]);
    v.w = fmaf(dcy, v.w, S[3 * kN]);
  }
}

}  // namespace fused
}  // namespace ssd

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
#include <stdlib.h>

#include <algorithm>
#include <atomic>
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

// bf16 tensor [d3][d2][d1][d0] (d0 contiguous, d1 rows d0 apart, d2 = tokens
// st.t elements apart, d3 = batch rows st.b apart); box = 64 x 1 x 128 x 1
// with the 128-byte swizzle, i.e. one [128 rows][64] operand block per copy;
// rows past d2 (the sequence end) are filled with zeros.
bool make_map(CUtensorMap* m, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
              uint64_t d3, TokStride st) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {d0, d1, d2, d3};
  cuuint64_t strides[3] = {d0 * 2, (cuuint64_t)st.t * 2, (cuuint64_t)st.b * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
             es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// per device; host threads may launch concurrently
int sm_count() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int n = cached[dev].load(std::memory_order_relaxed);
  if (n == 0) {
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    n = n > 0 ? n : 148;
    cached[dev].store(n, std::memory_order_relaxed);
  }
  return n;
}

// the shared-memory opt-in is a property of each kernel on each device
template <typename K>
cudaError_t ensure_smem(K kernel, size_t smem, int which) {
  static std::atomic<bool> done[8][64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const bool known = dev >= 0 && dev < 64;
  if (known && done[which][dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e == cudaSuccess && known) done[which][dev].store(true, std::memory_order_release);
  return e;
}

// Segment states on tensor cores (the pre-pass, or the chunk-state stage
// with one chunk per segment).  pa: the launch's Params with items, nseg,
// seg_chunks, ticket, seg_states and seg_decay set.
// pa.dt / pa.cs / pa.seg: stage 1's outputs (the kernel reads them, never the raw dt).
cudaError_t launch_segstate(const CUtensorMap& mx, const CUtensorMap& mb, const fused::Params& pa,
                            cudaStream_t st) {
  const size_t smem = sizeof(fused::SegSmem) + 1024;
  cudaError_t e = ensure_smem(fused::ssd_segstate_kernel, smem, 2);
  if (e != cudaSuccess) return e;
  const long long grid = std::min<long long>(pa.items, sm_count());
  fused::ssd_segstate_kernel<<<(unsigned)grid, fused::kSThreads, smem, st>>>(mx, mb, pa);
  return cudaGetLastError();
}

// control words of the stand-alone chunk-state and chunk-scan stages, which
// have no workspace: [0] and [2] ticket counters, [1] error word (cleared
// before each launch; the hand-off flags after them are not used there)
__device__ int g_stage_ctrl[64];

}  // namespace

bool fused_eligible(const Dims& d, bool bf16) {
  // TMA: token and batch strides of x, z, B, C multiples of 16 bytes (8 bf16
  // elements), positive and below 2^39 elements; dt read as bf16 pairs: even strides
  auto tma_ok = [](const TokStride& s) {
    return s.b > 0 && s.t > 0 && s.b % 8 == 0 && s.t % 8 == 0 && s.b < (1LL << 39) &&
           s.t < (1LL << 39);
  };
  return bf16 && d.headdim == fused::kP && d.dstate == fused::kN &&
         (d.chunk == 128 || d.chunk == 256) && (d.nheads / d.ngroups) % fused::kNH == 0 &&
         d.seqlen <= (int64_t)1 << 30 && tma_ok(d.sx) && tma_ok(d.sz) && tma_ok(d.sB) &&
         tma_ok(d.sC) && d.sdt.b % 2 == 0 && d.sdt.t % 2 == 0;
}

size_t fused_ctrl_ints(const Dims& d) { return 64 + (size_t)d.batch * d.nheads; }

cudaError_t launch_fused(const __nv_bfloat16* x, const __nv_bfloat16* Bm,
                         const __nv_bfloat16* Cm, const FusedVectors& v, const float* D,
                         const __nv_bfloat16* z, const float* init, float* final_states,
                         __nv_bfloat16* out, float* slots, int* ctrl, const Dims& d,
                         cudaStream_t st) {
  CUtensorMap mx, mb, mc, mz, mo;
  const int64_t hp = (int64_t)d.nheads * fused::kP;
  const TokStride dense_out = {d.seqlen * hp, hp};
  if (!make_map(&mx, x, fused::kP, d.nheads, d.seqlen, d.batch, d.sx) ||
      !make_map(&mb, Bm, fused::kN, d.ngroups, d.seqlen, d.batch, d.sB) ||
      !make_map(&mc, Cm, fused::kN, d.ngroups, d.seqlen, d.batch, d.sC) ||
      !make_map(&mo, out, fused::kP, d.nheads, d.seqlen, d.batch, dense_out))
    return cudaErrorInvalidValue;
  if (z && !make_map(&mz, z, fused::kP, d.nheads, d.seqlen, d.batch, d.sz))
    return cudaErrorInvalidValue;
  if (!z) mz = mx;   // never used
  // (stage 4 on its own uses no hand-off flags: the first 64 words only)
  cudaError_t e = cudaMemsetAsync(
      ctrl, 0, (v.prev_states ? 64 : fused_ctrl_ints(d)) * sizeof(int), st);
  if (e != cudaSuccess) return e;
  fused::Params p;
  p.dt_raw = v.dt_raw;
  p.sdt_b = d.sdt.b;
  p.sdt_t = d.sdt.t;
  p.dt_bias = v.dt_bias;
  p.A = v.A;
  p.seq_idx = v.dt_raw ? v.seq_idx : nullptr;
  p.softplus = v.softplus;
  p.do_clamp = v.do_clamp;
  p.lo = v.lo;
  p.hi = v.hi;
  p.dt = v.dt;
  p.cs = v.cs;
  p.seg = v.dt_raw ? nullptr : v.seg;
  p.has_seg = v.dt_raw ? v.seq_idx != nullptr : v.seg != nullptr;
  p.D = D;
  p.z = z;
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
  // chunks per work item: the state stays in TMEM across a segment and is
  // handed on only between segments (a boundary costs about one sub-step);
  // segments are the longest that still give every SM about twelve items, so
  // that dynamic scheduling evens out the tail.  On the 2.7B shape (16 chunks,
  // 320 head pairs) 1: 0.317 ms, 2: 0.292, 3: 0.282, 4: 0.287, 6: 0.285, 8: 0.300
  const long long pairs = (long long)d.batch * (d.nheads / fused::kNH);
  int seg = 1;
  while (seg < d.nchunks &&
         pairs * ((d.nchunks + seg) / (seg + 1)) >= 12LL * sm_count())
    ++seg;
  // State pre-pass.  With fewer head pairs than SMs the segments of a pair
  // would run one after another through the hand-off and leave most SMs
  // idle (a 131k-token single sequence: 64 pairs, 512 chunks).  Instead
  // every segment's own state is computed first, all in parallel; a short
  // pass over the segments gives the state entering each one; the main
  // kernel then reads those and never waits for another CTA.  The three
  // passes use the chunk-state region of the workspace (segments of at
  // least 3 chunks, so that the two tables fit).
  bool prepass = pairs < sm_count() && d.nchunks >= 8;
  if (const char* ov = getenv("SSD_FUSED_PREPASS")) prepass = atoi(ov) != 0;   // test override
  if (prepass) seg = std::max(seg, std::min(3, d.nchunks));
  if (const char* ov = getenv("SSD_FUSED_SEGMENT_CHUNKS")) {   // tuning / test override
    const int v = atoi(ov);
    if (v >= 1 && v <= d.nchunks) seg = v;
  }
  if (v.prev_states) {   // stage 4 on its own: every chunk reads its entering state
    seg = 1;
    prepass = false;
  }
  p.seg_chunks = seg;
  p.items = pairs * ((d.nchunks + seg - 1) / seg);
  // any single wait gives up after 2 s; the time-out test shortens the limit
  // and asks for a hand-off flag value that is never reached
  p.wait_ns = fused::kWaitNs;
  p.lookback_extra = 0;
  if (const char* ov = getenv("SSD_FUSED_WAIT_NS")) {
    const long long v = atoll(ov);
    if (v > 0) p.wait_ns = (unsigned long long)v;
  }
  if (const char* ov = getenv("SSD_FUSED_TEST_STALL"))
    if (atoi(ov) == 1) p.lookback_extra = 1 << 24;
  // dt can be negative only without softplus (and no clamp to a non-negative
  // floor), or when the clamp's ceiling is negative; stage-1 outputs given
  // by the caller are taken as possibly negative
  const bool nonneg = v.dt_raw && (v.softplus ? (!v.do_clamp || v.hi >= 0.f)
                                              : (v.do_clamp && v.lo >= 0.f));
  p.ticket = ctrl;
  p.hin = v.prev_states;
  p.hin_dense = v.prev_states != nullptr;
  p.nseg = v.prev_states ? d.nchunks : 0;
  p.seg_states = p.seg_decay = nullptr;
  if (prepass && v.dt_raw && !(v.work_dt && v.work_cs && v.work_seg)) prepass = false;
  if (prepass) {
    const int nseg = (d.nchunks + seg - 1) / seg;
    const size_t pn = (size_t)fused::kP * fused::kN, bh = (size_t)d.batch * d.nheads;
    const size_t decay_floats = (bh * nseg + 63) / 64 * 64;
    if (seg < 2 || bh * nseg * 2 * pn + decay_floats > bh * (size_t)d.nchunks * pn) {
      prepass = false;   // the table would not fit (segments too short)
    } else {
      fused::Params pa = p;
      pa.items = pairs * nseg;
      pa.nseg = nseg;
      pa.ticket = ctrl + 2;
      pa.seg_states = slots;
      pa.seg_decay = slots + bh * nseg * pn;
      float* hin = pa.seg_decay + decay_floats;
      if (v.dt_raw) {   // stage 1 first: the segment-state kernel reads its outputs
        e = launch_dt_cumsum<__nv_bfloat16>(v.dt_raw, v.dt_bias, v.softplus, v.lo, v.hi,
                                            v.do_clamp, v.A, v.seq_idx, d, v.work_dt,
                                            v.work_cs, v.seq_idx ? v.work_seg : nullptr, st);
        if (e != cudaSuccess) return e;
        pa.dt_raw = nullptr;
        pa.seq_idx = nullptr;
        pa.dt = v.work_dt;
        pa.cs = v.work_cs;
        pa.seg = v.seq_idx ? v.work_seg : nullptr;
      }
      e = launch_segstate(mx, mb, pa, st);
      if (e != cudaSuccess) return e;
      const long long threads = (long long)bh * (fused::kP / 4) * fused::kN;
      fused::segment_passing_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, st>>>(
          pa.seg_states, pa.seg_decay, init, hin, (int)d.batch, d.nheads, nseg);
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
      p.hin = hin;
      p.nseg = nseg;
    }
  }
  const size_t smem = sizeof(fused::Smem) + 1024;
  e = nonneg ? ensure_smem(fused::ssd_fused_kernel<false>, smem, 0)
             : ensure_smem(fused::ssd_fused_kernel<true>, smem, 1);
  if (e != cudaSuccess) return e;
  const long long grid = std::min<long long>(p.items, sm_count());   // one CTA per SM
  if (nonneg)
    fused::ssd_fused_kernel<false><<<(unsigned)grid, fused::kThreads, smem, st>>>(mx, mb, mc, mz,
                                                                                 mo, p);
  else
    fused::ssd_fused_kernel<true><<<(unsigned)grid, fused::kThreads, smem, st>>>(mx, mb, mc, mz,
                                                                                mo, p);
  return cudaGetLastError();
}

cudaError_t launch_chunk_state_tc(const __nv_bfloat16* x, const __nv_bfloat16* Bm,
                                  const float* dt_out, const float* cs, const int32_t* seg,
                                  const Dims& d, float* states, cudaStream_t st) {
  CUtensorMap mx, mb;
  if (!make_map(&mx, x, fused::kP, d.nheads, d.seqlen, d.batch, d.sx) ||
      !make_map(&mb, Bm, fused::kN, d.ngroups, d.seqlen, d.batch, d.sB))
    return cudaErrorInvalidValue;
  int* ctrl = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ctrl), g_stage_ctrl);
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(ctrl, 0, sizeof(g_stage_ctrl), st);
  if (e != cudaSuccess) return e;
  fused::Params p = {};
  p.dt = dt_out;
  p.cs = cs;
  p.seg = seg;
  p.has_seg = seg != nullptr;
  p.L = d.seqlen;
  p.B = (int)d.batch;
  p.H = d.nheads;
  p.G = d.ngroups;
  p.Q = d.chunk;
  p.nc = d.nchunks;
  p.seg_chunks = 1;   // one chunk per segment: the chunk-local states
  p.nseg = d.nchunks;
  p.items = (long long)d.batch * (d.nheads / fused::kNH) * d.nchunks;
  p.wait_ns = fused::kWaitNs;
  p.ctrl = ctrl;
  p.ticket = ctrl + 2;
  p.seg_states = states;
  p.seg_decay = nullptr;
  return launch_segstate(mx, mb, p, st);
}

cudaError_t launch_chunk_scan_tc(const __nv_bfloat16* x, const __nv_bfloat16* Bm,
                                 const __nv_bfloat16* Cm, const float* dt_out, const float* cs,
                                 const int32_t* seg, const float* prev_states, const float* D,
                                 const __nv_bfloat16* z, const Dims& d, __nv_bfloat16* out,
                                 cudaStream_t st) {
  int* ctrl = nullptr;
  cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void**>(&ctrl), g_stage_ctrl);
  if (e != cudaSuccess) return e;
  FusedVectors v = {};
  v.dt = dt_out;
  v.cs = cs;
  v.seg = seg;
  v.prev_states = prev_states;
  return launch_fused(x, Bm, Cm, v, D, z, nullptr, nullptr, out, nullptr, ctrl, d, st);
}

int fused_status(int reset, cudaStream_t st, int* bits) {
  int h = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&h, fused::g_status, sizeof(int), 0,
                                            cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e == cudaSuccess && reset && h != 0) {
    static const int zero = 0;
    e = cudaMemcpyToSymbolAsync(fused::g_status, &zero, sizeof(int), 0, cudaMemcpyHostToDevice,
                                st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  }
  *bits = h;
  return e == cudaSuccess ? 0 : (int)e;
}

}  // namespace ssd
