// ssd_scan_fwd_host: the forward with host-resident tensors.  The batch is
// cut into slices of batch rows; each slice is copied in, scanned and copied
// out through one of two device staging buffers, on three streams (copy in,
// compute, copy out) ordered with events, so that the copies of neighbouring
// slices overlap the kernel of the current one and each other.  Declared in
// include/ssd_scan.h.
#include <stdio.h>

#include <mutex>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"

namespace {

constexpr int kBufs = 2;   // device staging buffers (slices in flight)

size_t up256(size_t v) { return (v + 255) / 256 * 256; }

// Byte sizes of one batch row of each per-row tensor.
struct RowBytes {
  size_t x, dt, bc, seq, st;
};

RowBytes row_bytes(int64_t L, int H, int P, int N, int G, ssd_dtype_t dtype) {
  const size_t e = dtype == SSD_DTYPE_BF16 ? 2 : 4;
  RowBytes r;
  r.x = (size_t)L * H * P * e;     // x, z, out
  r.dt = (size_t)L * H * e;
  r.bc = (size_t)L * G * N * e;    // B, C
  r.seq = (size_t)L * 4;
  r.st = (size_t)H * P * N * 4;    // initial / final states
  return r;
}

// Layout of the caller's device workspace: the per-head arrays, then per
// staging buffer the slice's tensors and its scan workspace.
struct HostLayout {
  size_t heads;   // dt_bias, A, D: H floats each, 256-byte aligned
  size_t x, z, out, dt, B, C, seq, init, fin, scan;   // offsets inside a buffer
  size_t scan_bytes, buf_bytes, total;
};

HostLayout host_layout(int64_t rows, int64_t L, int H, int P, int N, int G, int Q,
                       ssd_dtype_t dtype) {
  const RowBytes rb = row_bytes(L, H, P, N, G, dtype);
  HostLayout l;
  l.heads = 3 * up256((size_t)H * sizeof(float));
  size_t o = 0;
  l.x = o;    o = up256(o + rows * rb.x);
  l.z = o;    o = up256(o + rows * rb.x);
  l.out = o;  o = up256(o + rows * rb.x);
  l.dt = o;   o = up256(o + rows * rb.dt);
  l.B = o;    o = up256(o + rows * rb.bc);
  l.C = o;    o = up256(o + rows * rb.bc);
  l.seq = o;  o = up256(o + rows * rb.seq);
  l.init = o; o = up256(o + rows * rb.st);
  l.fin = o;  o = up256(o + rows * rb.st);
  l.scan = o;
  l.scan_bytes = ssd_scan_workspace_bytes(rows, L, H, P, N, G, Q, dtype);
  l.buf_bytes = up256(o + l.scan_bytes);
  l.total = l.heads + kBufs * l.buf_bytes;
  return l;
}

// about eight slices: short fill and drain of the pipeline (measured on the
// 2.7B shape: 1 row of 8 per slice 4.21 ms, 2 rows 4.35, 4 rows 4.66)
int64_t default_rows(int64_t batch) { return (batch + 7) / 8; }

// Streams and events of the pipeline, one set per device, created on first
// use; `lock` serialises the enqueueing of calls that share them.
struct Pipe {
  bool ready = false;
  cudaStream_t in = nullptr, comp = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in_done[kBufs] = {}, comp_done[kBufs] = {}, out_done[kBufs] = {};
  std::mutex lock;
};

Pipe g_pipes[64];

cudaError_t pipe_init(Pipe& pp) {
  if (pp.ready) return cudaSuccess;
  cudaError_t e = cudaSuccess;
  cudaStream_t* ss[3] = {&pp.in, &pp.comp, &pp.out};
  for (cudaStream_t* s : ss)
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(s, cudaStreamNonBlocking);
  cudaEvent_t* es[2] = {&pp.start, &pp.end};
  for (cudaEvent_t* ev : es)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  for (int i = 0; i < kBufs && e == cudaSuccess; ++i) {
    e = cudaEventCreateWithFlags(&pp.in_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pp.comp_done[i], cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pp.out_done[i], cudaEventDisableTiming);
  }
  if (e == cudaSuccess) pp.ready = true;
  return e;
}

}  // namespace

extern "C" {

size_t ssd_scan_host_workspace_bytes(int64_t batch, int64_t seqlen, int nheads, int headdim,
                                     int dstate, int ngroups, int chunk_size, ssd_dtype_t dtype,
                                     int64_t rows_per_slice) {
  if (ssd_scan_workspace_bytes(batch, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                               dtype) == 0)
    return 0;   // bad sizes
  int64_t rows = rows_per_slice > 0 ? rows_per_slice : default_rows(batch);
  if (rows > batch) rows = batch;
  return host_layout(rows, seqlen, nheads, headdim, dstate, ngroups, chunk_size, dtype).total;
}

int ssd_scan_fwd_host(const void* x, const void* dt, const float* dt_bias, int dt_softplus,
                      float dt_limit_lo, float dt_limit_hi, const float* A, const void* B,
                      const void* C, const float* D, const void* z, const float* initial_states,
                      const int32_t* seq_idx, int64_t batch, int64_t seqlen, int nheads,
                      int headdim, int dstate, int ngroups, int chunk_size, ssd_dtype_t dtype,
                      void* out, float* final_states, int64_t rows_per_slice, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (!x || !dt || !A || !B || !C || !out || !workspace)
    return ssd::set_error(SSD_ERR_NULL, "x, dt, A, B, C, out and workspace are required");
  const size_t need = ssd_scan_host_workspace_bytes(batch, seqlen, nheads, headdim, dstate,
                                                    ngroups, chunk_size, dtype, rows_per_slice);
  if (need == 0)
    return ssd::set_error(SSD_ERR_ARG, "bad sizes (see ssd_scan_workspace_bytes)");
  if (workspace_bytes < need) {
    char msg[128];
    snprintf(msg, sizeof(msg), "workspace of %zu bytes < %zu needed", workspace_bytes, need);
    return ssd::set_error(SSD_ERR_WORKSPACE, msg);
  }
  if (((uintptr_t)workspace & 255u) != 0)
    return ssd::set_error(SSD_ERR_ALIGN, "workspace must be 256-byte aligned");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= 64)
    return ssd::set_error(SSD_ERR_CUDA, "no current CUDA device");
  Pipe& pp = g_pipes[dev];
  std::lock_guard<std::mutex> guard(pp.lock);
  e = pipe_init(pp);
  if (e != cudaSuccess) return ssd::set_error(SSD_ERR_CUDA, cudaGetErrorString(e));

  const int64_t rows = rows_per_slice > 0 ? (rows_per_slice < batch ? rows_per_slice : batch)
                                          : default_rows(batch);
  const HostLayout lay = host_layout(rows, seqlen, nheads, headdim, dstate, ngroups, chunk_size,
                                     dtype);
  const RowBytes rb = row_bytes(seqlen, nheads, headdim, dstate, ngroups, dtype);
  char* ws = static_cast<char*>(workspace);
  const size_t hslot = up256((size_t)nheads * sizeof(float));
  float* d_bias = reinterpret_cast<float*>(ws);
  float* d_A = reinterpret_cast<float*>(ws + hslot);
  float* d_D = reinterpret_cast<float*>(ws + 2 * hslot);
  cudaStream_t user = static_cast<cudaStream_t>(stream);
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;

  // the pipeline starts after the caller's earlier work on `stream`
  e = cudaEventRecord(pp.start, user);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.in, pp.start, 0);
  const size_t hb = (size_t)nheads * sizeof(float);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_A, A, hb, h2d, pp.in);
  if (e == cudaSuccess && dt_bias) e = cudaMemcpyAsync(d_bias, dt_bias, hb, h2d, pp.in);
  if (e == cudaSuccess && D) e = cudaMemcpyAsync(d_D, D, hb, h2d, pp.in);

  const char* hx = static_cast<const char*>(x);
  const char* hdt = static_cast<const char*>(dt);
  const char* hB = static_cast<const char*>(B);
  const char* hC = static_cast<const char*>(C);
  const char* hz = static_cast<const char*>(z);
  const char* hinit = reinterpret_cast<const char*>(initial_states);
  const char* hseq = reinterpret_cast<const char*>(seq_idx);
  char* hout = static_cast<char*>(out);
  char* hfin = reinterpret_cast<char*>(final_states);
  int rc = SSD_OK;
  int64_t slice = 0;
  for (int64_t r0 = 0; r0 < batch && e == cudaSuccess && rc == SSD_OK; r0 += rows, ++slice) {
    const int64_t nr = batch - r0 < rows ? batch - r0 : rows;
    const int bi = (int)(slice % kBufs);
    char* buf = ws + lay.heads + bi * lay.buf_bytes;
    // copies in: once the slice that used this buffer before has been copied out
    if (slice >= kBufs) e = cudaStreamWaitEvent(pp.in, pp.out_done[bi], 0);
    auto in = [&](size_t off, const char* src, size_t row_bytes) {
      if (e == cudaSuccess && src)
        e = cudaMemcpyAsync(buf + off, src + r0 * row_bytes, nr * row_bytes, h2d, pp.in);
    };
    in(lay.x, hx, rb.x);
    in(lay.dt, hdt, rb.dt);
    in(lay.B, hB, rb.bc);
    in(lay.C, hC, rb.bc);
    in(lay.z, hz, rb.x);
    in(lay.seq, hseq, rb.seq);
    in(lay.init, hinit, rb.st);
    if (e == cudaSuccess) e = cudaEventRecord(pp.in_done[bi], pp.in);
    // the scan of the slice
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pp.comp, pp.in_done[bi], 0);
    if (e == cudaSuccess && slice >= kBufs) e = cudaStreamWaitEvent(pp.comp, pp.out_done[bi], 0);
    if (e == cudaSuccess) {
      rc = ssd_scan_fwd(buf + lay.x, buf + lay.dt, dt_bias ? d_bias : nullptr, dt_softplus,
                        dt_limit_lo, dt_limit_hi, d_A, buf + lay.B, buf + lay.C,
                        D ? d_D : nullptr, z ? buf + lay.z : nullptr,
                        initial_states ? reinterpret_cast<const float*>(buf + lay.init) : nullptr,
                        seq_idx ? reinterpret_cast<const int32_t*>(buf + lay.seq) : nullptr, nr,
                        seqlen, nheads, headdim, dstate, ngroups, chunk_size, dtype,
                        buf + lay.out,
                        final_states ? reinterpret_cast<float*>(buf + lay.fin) : nullptr,
                        buf + lay.scan, lay.scan_bytes, pp.comp);
    }
    if (e == cudaSuccess && rc == SSD_OK) e = cudaEventRecord(pp.comp_done[bi], pp.comp);
    // copies out
    if (e == cudaSuccess && rc == SSD_OK) e = cudaStreamWaitEvent(pp.out, pp.comp_done[bi], 0);
    if (e == cudaSuccess && rc == SSD_OK)
      e = cudaMemcpyAsync(hout + r0 * rb.x, buf + lay.out, nr * rb.x, d2h, pp.out);
    if (e == cudaSuccess && rc == SSD_OK && hfin)
      e = cudaMemcpyAsync(hfin + r0 * rb.st, buf + lay.fin, nr * rb.st, d2h, pp.out);
    if (e == cudaSuccess && rc == SSD_OK) e = cudaEventRecord(pp.out_done[bi], pp.out);
  }
  // `stream` continues once the last slice is copied out
  if (e == cudaSuccess && rc == SSD_OK) e = cudaEventRecord(pp.end, pp.out);
  if (e == cudaSuccess && rc == SSD_OK) e = cudaStreamWaitEvent(user, pp.end, 0);
  if (e != cudaSuccess || rc != SSD_OK) {
    // on failure part of the pipeline may already be queued: let the copies
    // that read or write the caller's host buffers and workspace finish
    // before the caller gets the error and may free them
    cudaStreamSynchronize(pp.in);
    cudaStreamSynchronize(pp.comp);
    cudaStreamSynchronize(pp.out);
    if (rc != SSD_OK) return rc;   // ssd_scan_fwd set the message
    return ssd::set_error(SSD_ERR_CUDA, cudaGetErrorString(e));
  }
  return SSD_OK;
}

}  // extern "C"
