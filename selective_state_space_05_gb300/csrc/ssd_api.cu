// C-ABI entry points of the SSD chunked-scan library: argument validation,
// workspace carving and the launch sequence.  Declared in include/ssd_scan.h.
#include <math.h>
#include <stdarg.h>

#include <algorithm>
#include <stdio.h>
#include <string.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"

namespace {

thread_local char g_err[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return code;
}

int cuda_fail(cudaError_t e, const char* where) {
  return fail(SSD_ERR_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return p == nullptr || ((uintptr_t)p & 15u) == 0; }

size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Validates sizes shared by every entry point and fills Dims.  need_state:
// headdim/dstate/ngroups are used by this entry point.
int check_dims(int64_t batch, int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
               int chunk, bool need_state, ssd::Dims* d) {
  if (batch < 1 || seqlen < 1 || nheads < 1)
    return fail(SSD_ERR_ARG, "batch, seqlen and nheads must be >= 1 (got %lld, %lld, %d)",
                (long long)batch, (long long)seqlen, nheads);
  if (!(chunk == 16 || chunk == 32 || chunk == 64 || chunk == 128 || chunk == 256))
    return fail(SSD_ERR_UNSUPPORTED, "chunk_size must be one of 16, 32, 64, 128, 256 (got %d)",
                chunk);
  if (batch > 65535) return fail(SSD_ERR_UNSUPPORTED, "batch > 65535");
  if (nheads > 65535) return fail(SSD_ERR_UNSUPPORTED, "nheads > 65535");
  if (need_state) {
    if (ngroups < 1 || nheads % ngroups != 0)
      return fail(SSD_ERR_ARG, "nheads (%d) must be a positive multiple of ngroups (%d)",
                  nheads, ngroups);
    if (!(headdim == 16 || headdim == 32 || headdim == 64 || headdim == 128))
      return fail(SSD_ERR_UNSUPPORTED, "headdim must be one of 16, 32, 64, 128 (got %d)",
                  headdim);
    if (dstate < 16 || dstate > 256 || dstate % 16 != 0)
      return fail(SSD_ERR_UNSUPPORTED, "dstate must be a multiple of 16 in [16, 256] (got %d)",
                  dstate);
  }
  const int64_t nc = (seqlen + chunk - 1) / chunk;
  if (nc * (int64_t)batch > 2147483647LL)
    return fail(SSD_ERR_UNSUPPORTED, "batch * nchunks too large");
  d->batch = batch;
  d->seqlen = seqlen;
  d->nheads = nheads;
  d->headdim = headdim;
  d->dstate = dstate;
  d->ngroups = ngroups;
  d->chunk = chunk;
  d->nchunks = (int)nc;
  // dense inputs unless the strided entry point sets other strides
  const int64_t hp = (int64_t)nheads * headdim, gn = (int64_t)ngroups * dstate;
  d->sx = {seqlen * hp, hp};
  d->sz = d->sx;
  d->sdt = {seqlen * nheads, nheads};
  d->sB = {seqlen * gn, gn};
  d->sC = d->sB;
  return SSD_OK;
}

int check_dtype(ssd_dtype_t t) {
  if (t != SSD_DTYPE_F32 && t != SSD_DTYPE_BF16) return fail(SSD_ERR_ARG, "unknown dtype %d", (int)t);
  return SSD_OK;
}

struct Workspace {
  int* ctrl;   // fused path: ticket counter, error word, hand-off flags
  float* dt;
  float* cs;
  int32_t* seg;
  float* states;
  float* cb;   // C B^T per (batch, chunk, group) for the fp32 tensor-core stages, or nullptr
  float* tg;   // B as chunk_state's pre-split tiles (fp32, dstate 128), or nullptr
  size_t bytes;
};

// Whether fp32 at these sizes takes the fp32 tensor-core chunk_scan, which
// reads C B^T computed once per group (the workspace then holds it).
bool fp32_shared_cb(const ssd::Dims& d) {
  return d.chunk == 128 && (d.headdim == 64 || d.headdim == 128) && d.dstate % 32 == 0 &&
         d.dstate <= 256;
}

Workspace carve(const ssd::Dims& d, void* base, bool with_cb = false) {
  const size_t nq = (size_t)d.batch * d.nheads * d.nchunks * d.chunk;
  const size_t sq = (size_t)d.batch * d.nchunks * d.chunk;
  const size_t st = (size_t)d.batch * d.nchunks * d.nheads * d.headdim * d.dstate;
  Workspace w;
  size_t off = 0;
  char* p = static_cast<char*>(base);
  w.ctrl = reinterpret_cast<int*>(p + off);
  off = round_up(off + ssd::fused_ctrl_ints(d) * sizeof(int), 256);
  w.dt = reinterpret_cast<float*>(p + off);
  off = round_up(off + nq * sizeof(float), 256);
  w.cs = reinterpret_cast<float*>(p + off);
  off = round_up(off + nq * sizeof(float), 256);
  w.seg = reinterpret_cast<int32_t*>(p + off);
  off = round_up(off + sq * sizeof(int32_t), 256);
  w.states = reinterpret_cast<float*>(p + off);
  off = round_up(off + st * sizeof(float), 256);
  w.cb = nullptr;
  w.tg = nullptr;
  if (with_cb) {
    w.cb = reinterpret_cast<float*>(p + off);
    off = round_up(off + (size_t)d.batch * d.nchunks * d.ngroups * d.chunk * d.chunk *
                             sizeof(float), 256);
    if (d.dstate == 128) {
      w.tg = reinterpret_cast<float*>(p + off);
      off = round_up(off + (size_t)d.batch * d.nchunks * d.ngroups * (d.chunk / 16) *
                               ssd::group_tile_floats() * sizeof(float), 256);
    }
  }
  w.bytes = off;
  return w;
}

int do_clamp_of(float lo, float hi) { return !(lo == 0.f && isinf(hi) && hi > 0.f); }

// bf16 shapes outside the fused kernel that the fp32 tensor-core stages take
// run there, on fp32 copies of x, B, C and z (exact) made in the workspace,
// with out computed in fp32 and rounded to bf16 once (d: the caller's sizes).
bool bf16_via_fp32(const ssd::Dims& d) {
  return !ssd::fused_eligible(d, true) && (d.headdim == 64 || d.headdim == 128) &&
         d.dstate % 32 == 0 && d.dstate <= 256 && (d.chunk == 128 || d.chunk == 256);
}

// The fp32 copies, after the workspace regions that end at `end`: x, z and
// out [B, L, H, P], B and C [B, L, G, N], dense.
struct Copies {
  float *x, *z, *B, *C, *out;
  size_t bytes;
};
Copies copies_carve(const ssd::Dims& d, size_t end, void* base) {
  const size_t xs = (size_t)d.batch * d.seqlen * d.nheads * d.headdim;
  const size_t bs = (size_t)d.batch * d.seqlen * d.ngroups * d.dstate;
  char* p = static_cast<char*>(base);
  size_t off = round_up(end, 256);
  Copies c;
  auto take = [&](size_t elems) {
    float* at = reinterpret_cast<float*>(p + off);
    off = round_up(off + elems * sizeof(float), 256);
    return at;
  };
  c.x = take(xs);
  c.z = take(xs);
  c.out = take(xs);
  c.B = take(bs);
  c.C = take(bs);
  c.bytes = off;
  return c;
}

// bf16 rows of `row` elements, one per (batch, token) with token strides s
// (elements), into dense fp32; kVec: 8 elements per step (16-byte loads,
// strides and row multiples of 8).
template <bool kVec>
__global__ void __launch_bounds__(256) bf16_rows_to_f32_kernel(const __nv_bfloat16* __restrict__ src,
                                                               ssd::TokStride s, int64_t L, int row,
                                                               int64_t rows, float* __restrict__ dst) {
  constexpr int V = kVec ? 8 : 1;
  const int per = row / V;
  const int64_t total = rows * per;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / per, b = r / L, t = r % L;
    const int k = (int)(i % per) * V;
    const __nv_bfloat16* sp = src + ssd::toff(s, b, t) + k;
    float* dp = dst + r * row + k;
    if constexpr (kVec) {
      const uint4 v = *reinterpret_cast<const uint4*>(sp);
      const uint32_t w[4] = {v.x, v.y, v.z, v.w};
      float f[8];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        f[2 * u] = __uint_as_float(w[u] << 16);
        f[2 * u + 1] = __uint_as_float(w[u] & 0xFFFF0000u);
      }
      *reinterpret_cast<float4*>(dp) = make_float4(f[0], f[1], f[2], f[3]);
      *reinterpret_cast<float4*>(dp + 4) = make_float4(f[4], f[5], f[6], f[7]);
    } else {
      *dp = __bfloat162float(*sp);
    }
  }
}

// dense fp32 -> dense bf16 (round to nearest even), 8 elements per step
__global__ void __launch_bounds__(256) f32_to_bf16_rows_kernel(const float* __restrict__ src,
                                                               int64_t n8, __nv_bfloat16* __restrict__ dst) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8;
       i += (int64_t)gridDim.x * blockDim.x) {
    const float4 a = *reinterpret_cast<const float4*>(src + 8 * i);
    const float4 c = *reinterpret_cast<const float4*>(src + 8 * i + 4);
    __nv_bfloat162 o[4] = {__floats2bfloat162_rn(a.x, a.y), __floats2bfloat162_rn(a.z, a.w),
                           __floats2bfloat162_rn(c.x, c.y), __floats2bfloat162_rn(c.z, c.w)};
    *reinterpret_cast<uint4*>(dst + 8 * i) = *reinterpret_cast<const uint4*>(o);
  }
}

unsigned grid_for(int64_t n) {
  return (unsigned)std::min<int64_t>((n + 255) / 256, (int64_t)152 * 64);
}

// One bf16 tensor of rows (batch, token) into its dense fp32 copy.
cudaError_t rows_to_f32(const void* src, ssd::TokStride s, const ssd::Dims& d, int row, float* dst,
                        cudaStream_t st) {
  const int64_t rows = d.batch * d.seqlen;
  const bool vec = row % 8 == 0 && s.b % 8 == 0 && s.t % 8 == 0;
  if (vec)
    bf16_rows_to_f32_kernel<true><<<grid_for(rows * (row / 8)), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(src), s, d.seqlen, row, rows, dst);
  else
    bf16_rows_to_f32_kernel<false><<<grid_for(rows * row), 256, 0, st>>>(
        static_cast<const __nv_bfloat16*>(src), s, d.seqlen, row, rows, dst);
  return cudaGetLastError();
}

// The chunk length the forward's stages run at.  fp32 at chunk 256 runs them
// at 128 tokens when the headdim / dstate are ones the fp32 tensor-core
// stages take: the scan does not depend on the chunk length (only its
// rounding does), and those stages are built for 128-token chunks.
ssd::Dims fwd_dims(const ssd::Dims& d, ssd_dtype_t dtype) {
  ssd::Dims e = d;
  const bool tc = (d.headdim == 64 || d.headdim == 128) && d.dstate % 32 == 0 && d.dstate <= 256;
  const bool f32 = dtype == SSD_DTYPE_F32 || (dtype == SSD_DTYPE_BF16 && bf16_via_fp32(d));
  if (f32 && d.chunk == 256 && tc) {
    e.chunk = 128;
    e.nchunks = (int)((d.seqlen + 127) / 128);
  }
  return e;
}

}  // namespace

namespace ssd {
// Records an error message for ssd_last_error() from another translation unit.
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }

// The forward's workspace without the fp32 copies of bf16 inputs (the least
// a call takes: with less room for the copies it runs the bf16 stage
// kernels); 0 for invalid sizes.
size_t fwd_workspace_bytes_least(int64_t batch, int64_t seqlen, int nheads, int headdim,
                                 int dstate, int ngroups, int chunk_size, int dtype_in) {
  const ssd_dtype_t dtype = static_cast<ssd_dtype_t>(dtype_in);
  ssd::Dims d;
  if (check_dtype(dtype) != SSD_OK) return 0;
  if (check_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, true, &d) != SSD_OK)
    return 0;
  if (dtype == SSD_DTYPE_BF16) return carve(d, nullptr, false).bytes;
  const ssd::Dims e = fwd_dims(d, dtype);
  return carve(e, nullptr, fp32_shared_cb(e)).bytes;
}
}  // namespace ssd

extern "C" {

int ssd_abi_version(void) { return SSD_ABI_VERSION; }

const char* ssd_last_error(void) { return g_err; }

int ssd_scan_status(int reset, void* stream) {
  g_err[0] = 0;
  int bits = 0;
  int e = ssd::fused_status(reset, static_cast<cudaStream_t>(stream), &bits);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "ssd_scan_status");
  int bits32 = 0;
  e = ssd::tc32_status(reset, static_cast<cudaStream_t>(stream), &bits32);
  if (e != 0) return cuda_fail(static_cast<cudaError_t>(e), "ssd_scan_status");
  bits |= bits32;
  if (bits != 0)
    return fail(SSD_ERR_TIMEOUT,
                "a tensor-core scan launch gave up a bounded wait (error bits 0x%x: 1 barrier, "
                "2 state hand-off, 4 drain, 8 fp32 tensor-core stage); its outputs are not "
                "valid",
                bits);
  return SSD_OK;
}

size_t ssd_scan_workspace_bytes(int64_t batch, int64_t seqlen, int nheads, int headdim,
                                int dstate, int ngroups, int chunk_size, ssd_dtype_t dtype) {
  ssd::Dims d;
  if (check_dtype(dtype) != SSD_OK) return 0;
  if (check_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, true, &d) != SSD_OK)
    return 0;
  const ssd::Dims e = fwd_dims(d, dtype);
  const bool copies = dtype == SSD_DTYPE_BF16 && bf16_via_fp32(d);
  const size_t base = carve(e, nullptr, (dtype == SSD_DTYPE_F32 || copies) && fp32_shared_cb(e)).bytes;
  return copies ? copies_carve(e, base, nullptr).bytes : base;
}

int ssd_dt_cumsum(const void* dt, const float* dt_bias, int dt_softplus, float lo, float hi,
                  const float* A, const int32_t* seq_idx, int64_t batch, int64_t seqlen,
                  int nheads, int chunk_size, ssd_dtype_t dtype, float* dt_out,
                  float* dA_cumsum, int32_t* chunk_seg, void* stream) {
  g_err[0] = 0;
  ssd::Dims d;
  int rc = check_dtype(dtype);
  if (rc) return rc;
  rc = check_dims(batch, seqlen, nheads, 16, 16, 1, chunk_size, false, &d);
  if (rc) return rc;
  if (!dt || !A || !dt_out || !dA_cumsum)
    return fail(SSD_ERR_NULL, "dt, A, dt_out, dA_cumsum are required");
  if (seq_idx && !chunk_seg) return fail(SSD_ERR_NULL, "chunk_seg is required with seq_idx");
  if (!(lo <= hi)) return fail(SSD_ERR_ARG, "dt_limit lo > hi");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == SSD_DTYPE_F32)
    e = ssd::launch_dt_cumsum<float>(static_cast<const float*>(dt), dt_bias, dt_softplus, lo, hi,
                                     do_clamp_of(lo, hi), A, seq_idx, d, dt_out, dA_cumsum,
                                     chunk_seg, st);
  else
    e = ssd::launch_dt_cumsum<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(dt), dt_bias,
                                             dt_softplus, lo, hi, do_clamp_of(lo, hi), A, seq_idx,
                                             d, dt_out, dA_cumsum, chunk_seg, st);
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "dt_cumsum launch");
}

int ssd_chunk_state(const void* x, const void* B, const float* dt_out, const float* dA_cumsum,
                    const int32_t* chunk_seg, int64_t batch, int64_t seqlen, int nheads,
                    int headdim, int dstate, int ngroups, int chunk_size, ssd_dtype_t dtype,
                    float* states, void* stream) {
  g_err[0] = 0;
  ssd::Dims d;
  int rc = check_dtype(dtype);
  if (rc) return rc;
  rc = check_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, true, &d);
  if (rc) return rc;
  if (!x || !B || !dt_out || !dA_cumsum || !states)
    return fail(SSD_ERR_NULL, "x, B, dt_out, dA_cumsum, states are required");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == SSD_DTYPE_F32)
    e = ssd::launch_chunk_state<float>(static_cast<const float*>(x), static_cast<const float*>(B),
                                       dt_out, dA_cumsum, chunk_seg, d, states, st);
  else if (ssd::fused_eligible(d, true)) {   // tensor cores for the Mamba-2 shapes
    const void* ptrs[] = {x, B, dt_out, dA_cumsum, chunk_seg, states};
    for (const void* p : ptrs)
      if (!aligned16(p)) return fail(SSD_ERR_ALIGN, "every pointer must be 16-byte aligned");
    e = ssd::launch_chunk_state_tc(static_cast<const __nv_bfloat16*>(x),
                                   static_cast<const __nv_bfloat16*>(B), dt_out, dA_cumsum,
                                   chunk_seg, d, states, st);
  } else
    e = ssd::launch_chunk_state<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(x),
                                               static_cast<const __nv_bfloat16*>(B), dt_out,
                                               dA_cumsum, chunk_seg, d, states, st);
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "chunk_state launch");
}

int ssd_state_passing(float* states, const float* dA_cumsum, const int32_t* chunk_seg,
                      const float* initial_states, float* final_states, int64_t batch,
                      int64_t seqlen, int nheads, int headdim, int dstate, int chunk_size,
                      void* stream) {
  g_err[0] = 0;
  ssd::Dims d;
  int rc = check_dims(batch, seqlen, nheads, headdim, dstate, 1, chunk_size, true, &d);
  if (rc) return rc;
  if (!states || !dA_cumsum) return fail(SSD_ERR_NULL, "states and dA_cumsum are required");
  if (!aligned16(states) || !aligned16(initial_states) || !aligned16(final_states))
    return fail(SSD_ERR_ALIGN, "states, initial_states, final_states must be 16-byte aligned");
  cudaError_t e = ssd::launch_state_passing(states, dA_cumsum, chunk_seg, initial_states,
                                            final_states, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "state_passing launch");
}

int ssd_chunk_scan(const void* x, const void* B, const void* C, const float* dt_out,
                   const float* dA_cumsum, const int32_t* chunk_seg, const float* prev_states,
                   const float* D, const void* z, int64_t batch, int64_t seqlen, int nheads,
                   int headdim, int dstate, int ngroups, int chunk_size, ssd_dtype_t dtype,
                   void* out, void* stream) {
  g_err[0] = 0;
  ssd::Dims d;
  int rc = check_dtype(dtype);
  if (rc) return rc;
  rc = check_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, true, &d);
  if (rc) return rc;
  if (!x || !B || !C || !dt_out || !dA_cumsum || !prev_states || !out)
    return fail(SSD_ERR_NULL, "x, B, C, dt_out, dA_cumsum, prev_states, out are required");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (dtype == SSD_DTYPE_BF16 && ssd::fused_eligible(d, true)) {   // tensor cores
    const void* ptrs[] = {x, B, C, z, out, dt_out, dA_cumsum, chunk_seg, prev_states};
    for (const void* p : ptrs)
      if (!aligned16(p)) return fail(SSD_ERR_ALIGN, "every pointer must be 16-byte aligned");
    e = ssd::launch_chunk_scan_tc(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(B),
        static_cast<const __nv_bfloat16*>(C), dt_out, dA_cumsum, chunk_seg, prev_states, D,
        static_cast<const __nv_bfloat16*>(z), d, static_cast<__nv_bfloat16*>(out), st);
    return e == cudaSuccess ? SSD_OK : cuda_fail(e, "chunk_scan launch");
  }
  if (dtype == SSD_DTYPE_F32)
    e = ssd::launch_chunk_scan<float>(
        static_cast<const float*>(x), static_cast<const float*>(B), static_cast<const float*>(C),
        dt_out, dA_cumsum, chunk_seg, prev_states, D, static_cast<const float*>(z), d,
        static_cast<float*>(out), st);
  else
    e = ssd::launch_chunk_scan<__nv_bfloat16>(
        static_cast<const __nv_bfloat16*>(x), static_cast<const __nv_bfloat16*>(B),
        static_cast<const __nv_bfloat16*>(C), dt_out, dA_cumsum, chunk_seg, prev_states, D,
        static_cast<const __nv_bfloat16*>(z), d, static_cast<__nv_bfloat16*>(out), st);
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "chunk_scan launch");
}

size_t ssd_scan_workspace_bytes_min(int64_t batch, int64_t seqlen, int nheads, int headdim,
                                    int dstate, int ngroups, int chunk_size, ssd_dtype_t dtype) {
  return ssd::fwd_workspace_bytes_least(batch, seqlen, nheads, headdim, dstate, ngroups,
                                        chunk_size, dtype);
}

int ssd_chunk_fused(const void* x, const void* B, const void* C, const float* dt_out,
                    const float* dA_cumsum, const int32_t* chunk_seg, const float* D,
                    const void* z, const float* initial_states, int64_t batch, int64_t seqlen,
                    int nheads, int headdim, int dstate, int ngroups, int chunk_size,
                    ssd_dtype_t dtype, void* out, float* final_states, void* workspace,
                    size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  ssd::Dims d;
  int rc = check_dtype(dtype);
  if (rc) return rc;
  rc = check_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, true, &d);
  if (rc) return rc;
  if (!ssd::fused_eligible(d, dtype == SSD_DTYPE_BF16))
    return fail(SSD_ERR_UNSUPPORTED,
                "ssd_chunk_fused needs bf16, headdim 64, dstate 128, chunk_size 128 or 256 and an "
                "even number of heads per group");
  if (!x || !B || !C || !dt_out || !dA_cumsum || !out || !workspace)
    return fail(SSD_ERR_NULL, "x, B, C, dt_out, dA_cumsum, out and workspace are required");
  const void* ptrs[] = {x, B, C, z, out, initial_states, final_states, workspace, dt_out,
                        dA_cumsum, chunk_seg};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(SSD_ERR_ALIGN, "every pointer must be 16-byte aligned");
  const size_t need = carve(d, nullptr).bytes;
  if (workspace_bytes < need)
    return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  Workspace w = carve(d, workspace);
  using bf = __nv_bfloat16;
  ssd::FusedVectors v = {};
  v.dt = dt_out;
  v.cs = dA_cumsum;
  v.seg = chunk_seg;
  cudaError_t e = ssd::launch_fused(
      static_cast<const bf*>(x), static_cast<const bf*>(B), static_cast<const bf*>(C), v, D,
      static_cast<const bf*>(z), initial_states, final_states, static_cast<bf*>(out), w.states,
      w.ctrl, d, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "chunk_fused launch");
}

}  // extern "C"

namespace {

// The forward on validated sizes (and strides): workspace, dispatch, launches.
int scan_fwd_run(const ssd::Dims& d_in, const void* x, const void* dt, const float* dt_bias,
                 int dt_softplus, float dt_limit_lo, float dt_limit_hi, const float* A,
                 const void* B, const void* C, const float* D, const void* z,
                 const float* initial_states, const int32_t* seq_idx, ssd_dtype_t dtype,
                 void* out, float* final_states, void* workspace, size_t workspace_bytes,
                 void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // bf16 through the fp32 stages on fp32 copies, unless a caller's workspace
  // has no room for the copies (the bf16 stage kernels then run)
  bool copies = dtype == SSD_DTYPE_BF16 && bf16_via_fp32(d_in);
  ssd::Dims d = fwd_dims(d_in, dtype);
  bool with_cb = (dtype == SSD_DTYPE_F32 || copies) && fp32_shared_cb(d);
  size_t need = carve(d, nullptr, with_cb).bytes;
  if (copies) {
    const size_t with_copies = copies_carve(d, need, nullptr).bytes;
    if (workspace != nullptr && workspace_bytes < with_copies) {
      copies = false;
      d = d_in;
      with_cb = false;
      need = carve(d, nullptr, false).bytes;
    } else {
      need = with_copies;
    }
  }
  void* base = workspace;
  bool owned = false;
  if (base == nullptr) {
    cudaError_t e = cudaMallocAsync(&base, need, st);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(workspace)");
    owned = true;
  } else if (workspace_bytes < need) {
    return fail(SSD_ERR_WORKSPACE, "workspace of %zu bytes < %zu needed", workspace_bytes, need);
  }
  Workspace w = carve(d, base, with_cb);
  int32_t* seg = seq_idx ? w.seg : nullptr;
  const int clamp = do_clamp_of(dt_limit_lo, dt_limit_hi);
  cudaError_t e = cudaSuccess;
  if (dtype == SSD_DTYPE_F32 || copies) {
    const float* xf = static_cast<const float*>(x);
    const float* Bf = static_cast<const float*>(B);
    const float* Cf = static_cast<const float*>(C);
    const float* zf = static_cast<const float*>(z);
    float* of = static_cast<float*>(out);
    ssd::Dims df = d;   // the fp32 operands' layout
    if (copies) {       // dense fp32 copies of the bf16 x, B, C, z
      const Copies cp = copies_carve(d, w.bytes, base);
      const int hp = d.nheads * d.headdim, gn = d.ngroups * d.dstate;
      e = rows_to_f32(x, d.sx, d, hp, cp.x, st);
      if (e == cudaSuccess) e = rows_to_f32(B, d.sB, d, gn, cp.B, st);
      if (e == cudaSuccess) e = rows_to_f32(C, d.sC, d, gn, cp.C, st);
      if (e == cudaSuccess && z) e = rows_to_f32(z, d.sz, d, hp, cp.z, st);
      xf = cp.x;
      Bf = cp.B;
      Cf = cp.C;
      zf = z ? cp.z : nullptr;
      of = cp.out;
      df.sx = df.sz = {d.seqlen * hp, (int64_t)hp};
      df.sB = df.sC = {d.seqlen * gn, (int64_t)gn};
    }
    if (e == cudaSuccess)
      e = copies ? ssd::launch_dt_cumsum<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(dt),
                                                        dt_bias, dt_softplus, dt_limit_lo,
                                                        dt_limit_hi, clamp, A, seq_idx, d, w.dt,
                                                        w.cs, seg, st)
                 : ssd::launch_dt_cumsum<float>(static_cast<const float*>(dt), dt_bias,
                                                dt_softplus, dt_limit_lo, dt_limit_hi, clamp, A,
                                                seq_idx, d, w.dt, w.cs, seg, st);
    // chunk_state with B pre-split once per group where it runs on tensor cores
    const bool tg = w.tg != nullptr && ssd::chunk_state_tc32_fits(xf, Bf, df);
    if (e == cudaSuccess && tg)
      e = ssd::launch_group_tiles_tc32(Bf, df.sB, df.ngroups, df.batch, df.seqlen, df.nchunks,
                                       w.tg, st);
    if (e == cudaSuccess)
      e = tg ? ssd::launch_chunk_state_tc32(xf, Bf, w.dt, w.cs, seg, df, w.states, st, w.tg)
             : ssd::launch_chunk_state<float>(xf, Bf, w.dt, w.cs, seg, df, w.states, st);
    if (e == cudaSuccess)
      e = ssd::launch_state_passing(w.states, w.cs, seg, initial_states, final_states, df, st);
    // C B^T once per (batch, chunk, group) where chunk_scan runs on tensor cores
    const bool cb = w.cb != nullptr && ssd::cb_tc32_fits(Bf, Cf, df) &&
                    ssd::chunk_scan_tc32_fits(xf, Bf, Cf, zf, df);
    if (e == cudaSuccess && cb) e = ssd::launch_cb_tc32(Bf, Cf, df, w.cb, nullptr, st);
    if (e == cudaSuccess)
      e = cb ? ssd::launch_chunk_scan_tc32(xf, Bf, Cf, w.dt, w.cs, seg, w.states, D, zf, df, of,
                                           st, 0, w.cb, 0)
             : ssd::launch_chunk_scan<float>(xf, Bf, Cf, w.dt, w.cs, seg, w.states, D, zf, df,
                                             of, st);
    if (e == cudaSuccess && copies) {   // out rounded to bf16 once
      const int64_t n8 = d.batch * d.seqlen * d.nheads * d.headdim / 8;
      f32_to_bf16_rows_kernel<<<grid_for(n8), 256, 0, st>>>(of, n8,
                                                            static_cast<__nv_bfloat16*>(out));
      e = cudaGetLastError();
    }
  } else {
    using bf = __nv_bfloat16;
    const bf* xb = static_cast<const bf*>(x);
    if (ssd::fused_eligible(d, true)) {   // all four stages in one kernel
      ssd::FusedVectors v = {};
      v.dt_raw = static_cast<const bf*>(dt);
      v.dt_bias = dt_bias;
      v.A = A;
      v.seq_idx = seq_idx;
      v.softplus = dt_softplus;
      v.do_clamp = clamp;
      v.lo = dt_limit_lo;
      v.hi = dt_limit_hi;
      v.work_dt = w.dt;
      v.work_cs = w.cs;
      v.work_seg = w.seg;
      e = ssd::launch_fused(xb, static_cast<const bf*>(B), static_cast<const bf*>(C), v, D,
                            static_cast<const bf*>(z), initial_states, final_states,
                            static_cast<bf*>(out), w.states, w.ctrl, d, st);
    } else {
      e = ssd::launch_dt_cumsum<bf>(static_cast<const bf*>(dt), dt_bias, dt_softplus, dt_limit_lo,
                                    dt_limit_hi, clamp, A, seq_idx, d, w.dt, w.cs, seg, st);
      if (e == cudaSuccess)
        e = ssd::launch_chunk_state<bf>(xb, static_cast<const bf*>(B), w.dt, w.cs, seg, d,
                                        w.states, st);
      if (e == cudaSuccess)
        e = ssd::launch_state_passing(w.states, w.cs, seg, initial_states, final_states, d, st);
      if (e == cudaSuccess)
        e = ssd::launch_chunk_scan<bf>(xb, static_cast<const bf*>(B), static_cast<const bf*>(C),
                                       w.dt, w.cs, seg, w.states, D, static_cast<const bf*>(z),
                                       d, static_cast<bf*>(out), st);
    }
  }
  if (owned) {
    cudaError_t e2 = cudaFreeAsync(base, st);
    if (e == cudaSuccess) e = e2;
  }
  return e == cudaSuccess ? SSD_OK : cuda_fail(e, "ssd_scan_fwd launch");
}

int check_fwd_args(const void* x, const void* dt, const float* dt_bias, float lo, float hi,
                   const float* A, const void* B, const void* C, const float* D, const void* z,
                   const float* initial_states, const int32_t* seq_idx, void* out,
                   float* final_states, void* workspace) {
  if (!x || !dt || !A || !B || !C || !out)
    return fail(SSD_ERR_NULL, "x, dt, A, B, C and out are required");
  if (!(lo <= hi)) return fail(SSD_ERR_ARG, "dt_limit lo > hi");
  const void* ptrs[] = {x, dt, dt_bias, A, B, C, D, z, initial_states, seq_idx, out,
                        final_states, workspace};
  for (const void* p : ptrs)
    if (!aligned16(p)) return fail(SSD_ERR_ALIGN, "every pointer must be 16-byte aligned");
  return SSD_OK;
}

}  // namespace

extern "C" {

int ssd_scan_fwd(const void* x, const void* dt, const float* dt_bias, int dt_softplus,
                 float dt_limit_lo, float dt_limit_hi, const float* A, const void* B,
                 const void* C, const float* D, const void* z, const float* initial_states,
                 const int32_t* seq_idx, int64_t batch, int64_t seqlen, int nheads, int headdim,
                 int dstate, int ngroups, int chunk_size, ssd_dtype_t dtype, void* out,
                 float* final_states, void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  ssd::Dims d;
  int rc = check_dtype(dtype);
  if (rc) return rc;
  rc = check_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, true, &d);
  if (rc) return rc;
  rc = check_fwd_args(x, dt, dt_bias, dt_limit_lo, dt_limit_hi, A, B, C, D, z, initial_states,
                      seq_idx, out, final_states, workspace);
  if (rc) return rc;
  return scan_fwd_run(d, x, dt, dt_bias, dt_softplus, dt_limit_lo, dt_limit_hi, A, B, C, D, z,
                      initial_states, seq_idx, dtype, out, final_states, workspace,
                      workspace_bytes, stream);
}

int ssd_scan_fwd_strided(const void* x, ssd_stride_t x_stride, const void* dt,
                         ssd_stride_t dt_stride, const float* dt_bias, int dt_softplus,
                         float dt_limit_lo, float dt_limit_hi, const float* A, const void* B,
                         ssd_stride_t B_stride, const void* C, ssd_stride_t C_stride,
                         const float* D, const void* z, ssd_stride_t z_stride,
                         const float* initial_states, const int32_t* seq_idx, int64_t batch,
                         int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
                         int chunk_size, ssd_dtype_t dtype, void* out, float* final_states,
                         void* workspace, size_t workspace_bytes, void* stream) {
  g_err[0] = 0;
  ssd::Dims d;
  int rc = check_dtype(dtype);
  if (rc) return rc;
  rc = check_dims(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size, true, &d);
  if (rc) return rc;
  rc = check_fwd_args(x, dt, dt_bias, dt_limit_lo, dt_limit_hi, A, B, C, D, z, initial_states,
                      seq_idx, out, final_states, workspace);
  if (rc) return rc;
  const ssd_stride_t given[5] = {x_stride, dt_stride, B_stride, C_stride, z_stride};
  const char* names[5] = {"x", "dt", "B", "C", "z"};
  for (int i = 0; i < 5; ++i) {
    if (i == 4 && z == nullptr) continue;
    if (given[i].batch < 0 || given[i].token < 0 || given[i].batch > (1LL << 40) ||
        given[i].token > (1LL << 40))
      return fail(SSD_ERR_ARG, "%s strides must be in [0, 2^40] elements (got %lld, %lld)",
                  names[i], (long long)given[i].batch, (long long)given[i].token);
  }
  d.sx = {x_stride.batch, x_stride.token};
  d.sdt = {dt_stride.batch, dt_stride.token};
  d.sB = {B_stride.batch, B_stride.token};
  d.sC = {C_stride.batch, C_stride.token};
  if (z) d.sz = {z_stride.batch, z_stride.token};
  return scan_fwd_run(d, x, dt, dt_bias, dt_softplus, dt_limit_lo, dt_limit_hi, A, B, C, D, z,
                      initial_states, seq_idx, dtype, out, final_states, workspace,
                      workspace_bytes, stream);
}

}  // extern "C"
