// noalloc.cu -- decode entry point that needs no caller-provided workspace.
//
// Some callers cannot allocate device memory for us: an inference server that hands all
// free HBM to its KV-cache pool at start-up, a plugin that lives inside a host framework
// whose allocator owns the device, or a latency-critical loop where cudaMalloc's implicit
// synchronisation is not acceptable.  mla_attn_decode_noalloc serves them: the split-KV
// partial results that mla_attn_fwd keeps in the caller's workspace live here in a
// file-scope device array instead, so the call allocates nothing.
//
// The array is part of the library image: every GPU that loads the library holds it
// (kNoAllocScratchBytes) until the process exits.  All calls share it, so calls that
// overlap on the GPU (on different streams, or from different host threads) race on it;
// serialise them.  Each call overwrites every partial it later reads, so nothing in the
// array has to start at zero and stale contents from an earlier call are harmless.
#include <atomic>
#include <cmath>
#include <cstdint>

#include "kernels.h"
#include "mla_attn.h"

namespace mla {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;  // 32 MiB per device
constexpr int kMaxDevices = 64;

__device__ __align__(256) static uint8_t g_decode_scratch[kNoAllocScratchBytes];

// Device address of g_decode_scratch per device, looked up once with that device current.
std::atomic<uintptr_t> g_scratch_addr[kMaxDevices];

mla_status scratch_for_current_device(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MLA_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MLA_ERR_DEVICE;
  uintptr_t a = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (a == 0) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || ptr == nullptr)
      return MLA_ERR_CUDA;
    a = reinterpret_cast<uintptr_t>(ptr);
    g_scratch_addr[dev].store(a, std::memory_order_release);
  }
  *out = reinterpret_cast<uint8_t*>(a);
  return MLA_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_attn_decode_noalloc(const uint16_t* q_nope, const uint16_t* q_pe,
                                              const uint16_t* k_nope,
                                              const uint16_t* k_pe_shared, const uint16_t* v,
                                              const int32_t* kv_len, int B, int H, int Tk,
                                              float softmax_scale, uint16_t* out,
                                              int* device_status, void* cuda_stream) {
  if (!q_nope || !q_pe || !k_nope || !k_pe_shared || !v || !out) return MLA_ERR_NULL;
  if (B < 1 || H < 1 || Tk < 1 || B > 65535) return MLA_ERR_SHAPE;
  if ((int64_t)B * H * Tk * 128 > (int64_t(1) << 40)) return MLA_ERR_SHAPE;
  if (!aligned16(q_nope) || !aligned16(q_pe) || !aligned16(k_nope) || !aligned16(k_pe_shared) ||
      !aligned16(v) || !aligned16(out) || (reinterpret_cast<uintptr_t>(kv_len) & 3u) != 0 ||
      (reinterpret_cast<uintptr_t>(device_status) & 3u) != 0)
    return MLA_ERR_ALIGN;
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.0f)) return MLA_ERR_ARG;
  if (device_sm_count() <= 0) return MLA_ERR_DEVICE;

  // Same split plan as mla_attn_fwd's decode path, so the two give identical results.
  const DecodePlan pl = plan_decode(B, H, Tk, device_sm_count(), 0);
  const int chunk = pl.chunk, splits = pl.splits;
  const size_t rows = (size_t)B * H * splits;
  const size_t ml_bytes = (rows * 2 * sizeof(float) + 255) & ~(size_t)255;
  const size_t need = splits > 1 ? ml_bytes + rows * 128 * sizeof(float) : 0;
  if (need > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE;

  uint8_t* scratch = nullptr;
  const mla_status st = scratch_for_current_device(&scratch);
  if (st != MLA_OK) return st;

  DecodeArgs a{};
  a.q_nope = q_nope;
  a.q_pe = q_pe;
  a.k_nope = k_nope;
  a.k_pe = k_pe_shared;
  a.v = v;
  a.kv_len = kv_len;
  a.out = out;
  a.part_ml = reinterpret_cast<float*>(scratch);
  a.part_acc = reinterpret_cast<float*>(scratch + ml_bytes);
  a.status = device_status;
  a.B = B;
  a.H = H;
  a.Tk = Tk;
  a.chunk = chunk;
  a.splits = splits;
  a.kv_rows = Tk;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  return launch_decode(a, static_cast<cudaStream_t>(cuda_stream)) == cudaSuccess ? MLA_OK
                                                                                 : MLA_ERR_CUDA;
}
