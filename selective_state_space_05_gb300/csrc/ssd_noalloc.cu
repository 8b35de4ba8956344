// ssd_scan_fwd_noalloc: the scan forward for callers that cannot allocate
// device memory.  The scratch that ssd_scan_fwd would take from the caller or
// from cudaMallocAsync (processed dt, per-chunk cumsum and reset counts, chunk
// states) lives here in one file-scope device array instead.
#include <stdio.h>

#include "../../include/ssd_scan.h"
#include "ssd_common.cuh"

namespace {

// Fixed scratch, reserved in every GPU's memory when the library's module is
// loaded on that device and held until the process exits.
constexpr size_t kScratchBytes = SSD_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch in the current context.  In host code the name
// g_scratch is only a host-side stand-in; the real address comes from
// cudaGetSymbolAddress with the device current.  It is looked up on every
// call (cheap once the module is loaded), so that a context that was reset or
// re-created in between never gets a stale address.
int scratch_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_scratch);
  if (e != cudaSuccess || p == nullptr) {
    char m[256];
    snprintf(m, sizeof(m), "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    return ssd::set_error(SSD_ERR_CUDA, m);
  }
  *out = p;
  return SSD_OK;
}

}  // namespace

extern "C" {

int ssd_scan_fwd_noalloc(const void* x, const void* dt, const float* dt_bias, int dt_softplus,
                         float dt_limit_lo, float dt_limit_hi, const float* A, const void* B,
                         const void* C, const float* D, const void* z,
                         const float* initial_states, const int32_t* seq_idx, int64_t batch,
                         int64_t seqlen, int nheads, int headdim, int dstate, int ngroups,
                         int chunk_size, ssd_dtype_t dtype, void* out, float* final_states,
                         void* stream) {
  // (bf16 shapes outside the fused kernel run on the bf16 stage kernels when
  // the scratch has no room for fp32 copies of their inputs)
  const size_t need = ssd::fwd_workspace_bytes_least(batch, seqlen, nheads, headdim, dstate,
                                                     ngroups, chunk_size, dtype);
  if (need > kScratchBytes) {
    char m[256];
    snprintf(m, sizeof(m),
             "ssd_scan_fwd_noalloc: these sizes need %zu bytes of scratch but the static "
             "scratch holds %zu; use ssd_scan_fwd with a workspace",
             need, kScratchBytes);
    return ssd::set_error(SSD_ERR_WORKSPACE, m);
  }
  void* scratch = nullptr;
  int rc = scratch_address(&scratch);
  if (rc != SSD_OK) return rc;
  // need == 0 means invalid sizes: ssd_scan_fwd reports which one.  Nothing in
  // the scratch has to start at zero: every element a call reads is written
  // earlier in the same call.
  return ssd_scan_fwd(x, dt, dt_bias, dt_softplus, dt_limit_lo, dt_limit_hi, A, B, C, D, z,
                      initial_states, seq_idx, batch, seqlen, nheads, headdim, dstate, ngroups,
                      chunk_size, dtype, out, final_states, scratch, kScratchBytes, stream);
}

}  // extern "C"
