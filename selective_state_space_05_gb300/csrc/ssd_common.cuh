// Shared device helpers and the launcher interface between the C-ABI layer
// (ssd_api.cu) and the kernel files.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ssd {

constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f(float v);
template <> __device__ __forceinline__ float from_f<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// 2^x on the SFU (PTX ex2.approx, flush-to-zero).  Every exponential of the
// scan is exp(v), evaluated as 2^(v*log2 e); v <= 0 (a decay) whenever dt >= 0,
// and v > 0 only when the caller turns softplus off and passes negative dt
// (the state then grows; the result overflows only where the true value
// leaves the fp32 range).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Element strides between batch rows and between tokens of a
// [batch, seqlen, ...] input whose per-token part is dense (x, z: [nheads,
// headdim]; dt: [nheads]; B, C: [ngroups, dstate]).
struct TokStride {
  int64_t b, t;
};
__host__ __device__ __forceinline__ int64_t toff(const TokStride& s, int64_t b, int64_t t) {
  return b * s.b + t * s.t;
}

// Problem sizes as every launcher sees them, and the strides of the inputs
// (dense unless the caller gave others); out is always dense.
struct Dims {
  int64_t batch, seqlen;
  int nheads, headdim, dstate, ngroups, chunk;
  int nchunks;
  TokStride sx, sdt, sB, sC, sz;
  // heads that share one x row (x row of head h: h / xrep); 1 except where
  // the backward scans a per-group operand (B or C) in the place of x
  int xrep = 1;
};

// Launchers (return cudaGetLastError() of their launches).
template <typename T>
cudaError_t launch_dt_cumsum(const T* dt, const float* dt_bias, int softplus, float lo,
                             float hi, int do_clamp, const float* A, const int32_t* seq_idx,
                             const Dims& d, float* dt_out, float* cs, int32_t* seg,
                             cudaStream_t st);
template <typename T>
cudaError_t launch_chunk_state(const T* x, const T* B, const float* dt_out, const float* cs,
                               const int32_t* seg, const Dims& d, float* states,
                               cudaStream_t st);
cudaError_t launch_state_passing(float* states, const float* cs, const int32_t* seg,
                                 const float* init, float* final_states, const Dims& d,
                                 cudaStream_t st);
// strict = 1 leaves out the diagonal j = i of the intra-chunk sum (the
// backward's scans use that form; the forward always passes 0).
template <typename T>
cudaError_t launch_chunk_scan(const T* x, const T* B, const T* C, const float* dt_out,
                              const float* cs, const int32_t* seg, const float* prev,
                              const float* D, const T* z, const Dims& d, T* out,
                              cudaStream_t st, int strict = 0);

// Fused tensor-core kernel, bf16, headdim 64, dstate 128, chunk 128 or 256.
// Stages 2-4 always; stage 1 too when the per-token vectors are given raw
// (dt_raw set): then dt / cs / seg are not read.  ctrl: fused_ctrl_ints(d)
// ints of workspace, cleared by the launcher; slots: 2 * batch * nheads *
// headdim * dstate floats.
struct FusedVectors {
  const __nv_bfloat16* dt_raw;   // [B, L, H] raw dt, or null
  const float* dt_bias;          // [H] or null
  const float* A;                // [H] (with dt_raw)
  const int32_t* seq_idx;        // [B, L] or null (with dt_raw)
  int softplus, do_clamp;
  float lo, hi;
  const float* dt;               // stage-1 outputs (without dt_raw)
  const float* cs;
  const int32_t* seg;            // or null
  // workspace for stage 1's outputs (dt, cs [B, H, nc, Q]; seg [B, nc, Q]),
  // which the state pre-pass computes first when it runs from raw dt
  float* work_dt;
  float* work_cs;
  int32_t* work_seg;
  // stage 3's states entering every chunk ([B, nc, H, P, N]), or null: with
  // them the kernel takes each chunk's entering state from there (one chunk
  // per work item, no hand-off, no pre-pass) -- stage 4 on its own
  const float* prev_states;
};
bool fused_eligible(const Dims& d, bool bf16);
// Stage 2 (chunk states, [B, nc, H, P, N]) on tensor cores from stage 1's
// outputs, for the shapes fused_eligible accepts (bf16, headdim 64, dstate
// 128, chunk 128 / 256, an even number of heads per group).
cudaError_t launch_chunk_state_tc(const __nv_bfloat16* x, const __nv_bfloat16* B,
                                  const float* dt_out, const float* cs, const int32_t* seg,
                                  const Dims& d, float* states, cudaStream_t st);
// Stage 4 (chunk outputs) on tensor cores from stage 1's outputs and stage
// 3's prev_states, for the shapes fused_eligible accepts.
cudaError_t launch_chunk_scan_tc(const __nv_bfloat16* x, const __nv_bfloat16* B,
                                 const __nv_bfloat16* C, const float* dt_out, const float* cs,
                                 const int32_t* seg, const float* prev_states, const float* D,
                                 const __nv_bfloat16* z, const Dims& d, __nv_bfloat16* out,
                                 cudaStream_t st);
// fp32 stages 2 and 4 on the tensor cores (3xTF32, ssd_tc32.cu) for
// 128-token chunks, headdim 64 or 128; chunk_state also needs dstate 64 or
// 128 (one of the two 128), chunk_scan a dstate multiple of 32 up to 256.
// The fp32 SIMT launchers route there when *_fits holds (16-byte aligned
// rows; SSD_TC32=0 in the environment turns the route off).
bool chunk_state_tc32_fits(const float* x, const float* B, const Dims& d);
bool chunk_scan_tc32_fits(const float* x, const float* B, const float* C, const float* z,
                          const Dims& d);
// Tg: the 128-row per-group operand's split tiles from launch_group_tiles_tc32
// (B when dstate is 128; x, read through xrep, otherwise), or nullptr.
cudaError_t launch_chunk_state_tc32(const float* x, const float* B, const float* dtp,
                                    const float* cs, const int32_t* seg, const Dims& d,
                                    float* states, cudaStream_t st, const float* Tg = nullptr);
// A per-group operand Y [batch, seqlen, groups, 128] (token strides sY) as
// chunk_state's split A tiles: T holds batch x nchunks x groups x 8 slices of
// group_tile_floats() floats (128-token chunks).
constexpr int64_t group_tile_floats() { return 128 * 16 * 2; }
cudaError_t launch_group_tiles_tc32(const float* Y, TokStride sY, int groups, int64_t batch,
                                    int64_t seqlen, int nchunks, float* T, cudaStream_t st);
// Sg: C B^T of every (batch x chunk, group) computed beforehand by
// launch_cb_tc32 (nullptr: the kernel computes it itself); srev: read it for
// a time-reversed scan (chunk nc - 1 - c, indices 127 - i, 127 - j; pass the
// transposed copy there).
cudaError_t launch_chunk_scan_tc32(const float* x, const float* B, const float* C,
                                   const float* dtp, const float* cs, const int32_t* seg,
                                   const float* prev, const float* D, const float* z,
                                   const Dims& d, float* out, cudaStream_t st, int strict,
                                   const float* Sg = nullptr, int srev = 0);
// C B^T per (batch x chunk, group) into S [B][nc][G][128][128] fp32 (and its
// transpose into ST unless nullptr), for 128-token chunks, dstate a multiple
// of 16 up to 256.
bool cb_tc32_fits(const float* B, const float* C, const Dims& d);
cudaError_t launch_cb_tc32(const float* B, const float* C, const Dims& d, float* S, float* ST,
                           cudaStream_t st);
// Status bits of their bounded waits (8: a wait gave up), as fused_status.
int tc32_status(int reset, cudaStream_t st, int* bits);

// Device-wide status of the fused kernel's bounded waits: the error bits
// recorded since the last reset into *bits (0: none); synchronises st.
// Returns 0 or the cudaError_t of a failed copy.
int fused_status(int reset, cudaStream_t st, int* bits);
size_t fused_ctrl_ints(const Dims& d);
cudaError_t launch_fused(const __nv_bfloat16* x, const __nv_bfloat16* B, const __nv_bfloat16* C,
                         const FusedVectors& v, const float* D, const __nv_bfloat16* z,
                         const float* init, float* final_states, __nv_bfloat16* out,
                         float* slots, int* ctrl, const Dims& d, cudaStream_t st);

// Sets the per-thread message returned by ssd_last_error(); returns code.
int set_error(int code, const char* msg);

// The forward's workspace without the fp32 copies that bf16 shapes outside
// the fused kernel take when there is room (then the bf16 stage kernels run).
// (dtype: an ssd_dtype_t value)
size_t fwd_workspace_bytes_least(int64_t batch, int64_t seqlen, int nheads, int headdim,
                                 int dstate, int ngroups, int chunk_size, int dtype);

}  // namespace ssd
