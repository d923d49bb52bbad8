// rglru_forward_noalloc: the recurrence forward for callers that cannot allocate device
// memory.
//
// Who needs it: code that runs where cudaMalloc is off limits — inside a CUDA-graph capture
// region owned by someone else, under a fixed-budget memory pool or allocator that forbids
// new reservations, in a real-time inference loop that must not touch the allocator, or in a
// plugin that is handed only its input and output buffers.  Such a caller cannot provide the
// `saved` buffer that rglru_forward needs for its cross-chunk look-back scratch (flags,
// chunk aggregates and chunk-boundary states).
//
// What it does instead: the scratch lives in one file-scope device array of fixed size
// (RGLRU_NOALLOC_SCRATCH_BYTES, 16 MiB), created when the library is loaded on each GPU and
// held until the process exits.  Calls whose scratch would not fit are rejected with
// RGLRU_ERR_UNSUPPORTED.  Nothing here calls cudaMalloc, cudaFree or any allocating routine.
//
// Because the host cannot use the array's name as a device address, the first call on each
// device looks up the array's device address with cudaGetSymbolAddress (with that device
// current) and caches it; make that first call outside any stream capture.  Every call
// shares the one array: the part that must start at zero is cleared on the caller's stream
// at the start of each call, and two calls whose kernels overlap on the GPU (different
// streams without ordering between them) race on it.
#include <stdio.h>

#include <mutex>

#include "internal.h"

using namespace rglru;

namespace {

constexpr size_t kScratchBytes = RGLRU_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

rglru_status rglru_forward_noalloc(const rglru_shape* shape, const void* x, const void* lr,
                                   const void* li, const float* Lambda,
                                   const uint8_t* reset_mask, const int32_t* segment_pos,
                                   const float* h0, void* y, float* hT, rglru_stream stream) {
  Dims d;
  rglru_status st = make_dims(shape, &d);
  if (st != RGLRU_OK) return st;
  if (!req(x) || !req(lr) || !req(li) || !req(Lambda) || !req(y) || !opt(hT))
    return RGLRU_ERR_INVALID_ARG;
  if ((st = check_resets(d, reset_mask, segment_pos, h0)) != RGLRU_OK) return st;
  // bf16 goes through the fused scan kernel with the logits given (as rglru_forward does),
  // float32 through the CUDA-core scan
  const bool lg = logits_scan_supported(d);
  const size_t need = lg ? fused_fwd_layout(d).total : scan_layout(d, false).total;
  if (need > kScratchBytes) {
    fprintf(stderr,
            "librglru: rglru_forward_noalloc needs %zu bytes of look-back scratch for this "
            "shape; the static scratch holds %zu bytes (use rglru_forward with a caller "
            "buffer)\n",
            need, kScratchBytes);
    return RGLRU_ERR_UNSUPPORTED;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return cuda_status(e);
  if (lg)
    return cuda_status(launch_logits_fwd(d, x, lr, li, d.N, 1, Lambda, reset_mask, segment_pos,
                                         h0, y, hT, scratch, debug_spin_limit(),
                                         debug_drop_tile(), stream));
  const ScanFwdArgs a =
      fwd_args(d, x, lr, li, Lambda, reset_mask, segment_pos, h0, y, hT, scratch);
  e = cudaMemsetAsync(scratch, 0, a.L.zero_bytes, stream);
  if (e == cudaSuccess) e = launch_scan_fwd(a, d.io, d.io, d.mode == RGLRU_CANONICAL, stream);
  return cuda_status(e);
}

rglru_status rglru_forward_noalloc_status(rglru_stream stream) {
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) return cuda_status(e);
  uint32_t word = 0;
  e = cudaStreamSynchronize(stream);
  if (e == cudaSuccess) e = cudaMemcpy(&word, scratch, sizeof(word), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_status(e);
  return word ? RGLRU_ERR_TIMEOUT : RGLRU_OK;
}

}  // extern "C"
