// Verify + accept without any device allocation.
//
// The regular dflash_verify_accept runs on a context, and creating a context
// allocates device memory (ring, activations, the verify kernel's partial
// results). Some callers cannot do that: a host framework that hands out all
// device memory from its own pool and budget and forbids raw cudaMalloc, or a
// latency-critical loop that must never hit cudaMalloc's implicit
// device-wide synchronization. For them this file keeps the verify kernel's
// scratch (its per-chunk partial argmaxes, the "last CTA" ticket counter and
// a round-state record the kernel writes) in one statically sized
// __device__ array, so the call needs only the caller's own buffers.
#include <mutex>

#include "../../include/dflash.h"
#include "kernels.h"

namespace {

// Largest verify width and vocabulary the static scratch is sized for.
constexpr int kMaxBlockStatic = 64;
constexpr int kMaxVocabStatic = 1 << 20;
constexpr int kMaxChunks = kMaxVocabStatic / 8192;
constexpr size_t kPartials = (size_t)kMaxBlockStatic * kMaxChunks;
constexpr size_t kHeader = 256;                     // counter + round-state record
constexpr size_t kScratchBytes = kHeader + kPartials * (sizeof(float) + sizeof(int));

// Every GPU that loads the library holds this array (about 64 KB) until the
// process exits. All calls share it.
static __device__ __align__(256) unsigned char g_verify_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_dev[kMaxDevices] = {};

// Device address of the scratch on the current device. The symbol's name in
// host code is only a host-side stand-in, so the address is looked up with
// that device current. It is looked up again on every call made outside a
// stream capture (a device reset reloads the module, which can move the
// array); a call on a capturing stream uses the address found last.
int scratch_address(cudaStream_t st, void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    dfl::set_global_error("dflash_verify_accept_static: no usable current CUDA device");
    return DFLASH_ECUDA;
  }
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  e = cudaStreamIsCapturing(st, &cap);
  if (e != cudaSuccess) {
    dfl::set_global_error(cudaGetErrorString(e));
    return DFLASH_ECUDA;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_dev[dev] || cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_verify_scratch);
    if (e != cudaSuccess || !p) {
      dfl::set_global_error(cudaGetErrorString(e));
      return DFLASH_ECUDA;
    }
    g_scratch_dev[dev] = p;
  }
  *out = g_scratch_dev[dev];
  return DFLASH_OK;
}

}  // namespace

extern "C" int dflash_verify_accept_static(const void* target_logits, int32_t dtype, int32_t vocab,
                                           int32_t block, const int32_t* draft_ids, int32_t* tokens,
                                           int32_t* n, void* stream) {
  if (!target_logits || !draft_ids || !tokens || !n) {
    dfl::set_global_error("dflash_verify_accept_static: a pointer is NULL");
    return DFLASH_EINVAL;
  }
  if (dtype != DFLASH_F32 && dtype != DFLASH_BF16) {
    dfl::set_global_error("dflash_verify_accept_static: dtype must be DFLASH_F32 or DFLASH_BF16");
    return DFLASH_EINVAL;
  }
  if (block < 2 || block > kMaxBlockStatic || vocab < 2 || vocab > kMaxVocabStatic) {
    dfl::set_global_error("dflash_verify_accept_static: needs 2 <= block <= 64 and 2 <= vocab <= 1048576 "
                          "(the size of its static scratch)");
    return DFLASH_ERANGE;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  void* base = nullptr;
  int rc = scratch_address(st, &base);
  if (rc) return rc;
  auto* bytes = static_cast<unsigned char*>(base);
  unsigned* counter = reinterpret_cast<unsigned*>(bytes);
  dfl::RoundState* rs = reinterpret_cast<dfl::RoundState*>(bytes + 64);
  float* part_v = reinterpret_cast<float*>(bytes + kHeader);
  int* part_i = reinterpret_cast<int*>(bytes + kHeader + kPartials * sizeof(float));
  // The ticket counter must start at zero: clear it in case an earlier call
  // was cut short. Calls that overlap on the GPU share this array and race.
  cudaError_t e = cudaMemsetAsync(counter, 0, sizeof(unsigned), st);
  if (e == cudaSuccess) {
    dfl::VerifyArgs a{};
    a.L = target_logits; a.B = block; a.V = vocab; a.d = draft_ids; a.tokens = tokens; a.n = n;
    a.rs = rs; a.part_v = part_v; a.part_i = part_i; a.counter = counter;
    a.chunks = dfl::verify_chunks(vocab);
    e = dfl::launch_verify(dtype, a, st);
  }
  if (e != cudaSuccess) {
    dfl::set_global_error(cudaGetErrorString(e));
    return DFLASH_ECUDA;
  }
  return DFLASH_OK;
}
