// pva_forward_noalloc: the same attention as pva_forward for callers that
// must not allocate device memory at call time -- for example an inference
// runtime whose memory is fully planned ahead (a static arena or a memory
// governor that owns every byte), code running while another component holds
// the allocator, or a process that has to stay within a fixed device
// footprint.  pva_forward grows a per-stream workspace with cudaMalloc on
// first use; this entry point never calls cudaMalloc, cudaFree or any
// allocating library routine.  Its scratch (the scheduler's work lists, the
// decode kernel's split partials and completion counters, and a status word)
// lives in one file-scope device array of fixed size.  The array belongs to
// the library's device code: on each device it is bound when that code is
// loaded there (with CUDA's lazy module loading, at the first call that needs
// it) and those 4 MiB stay taken until the process exits.
//
// Consequences for callers:
//   * Every call on a device shares the one array.  Calls whose kernels
//     overlap on the GPU (different streams, or host threads without
//     ordering between them) race on it and produce wrong results; order such
//     calls (one stream, or events between streams).
//   * The array keeps what the last call left.  Everything that must start at
//     zero is cleared by each call itself: the decode completion counters by
//     the scheduler kernel, the internal status word by a memset at the start
//     of the call.
//   * Batches whose work lists need more than the fixed int region (roughly
//     B * (4 + kv_num_heads) int32 words above 1 MiB) are rejected with
//     PVA_ERR_UNSUPPORTED; decode split partials are limited to what fits in
//     the rest of the array (the scheduler picks fewer, larger splits when
//     needed).
//   * Without a caller status word the call latches its device-side errors
//     (malformed offsets, NULL tensors with a nonzero extent, a pipeline wait
//     that gave up) into a word inside the array that nothing reads back:
//     such a call leaves the output unwritten and the caller is not told.
//     Pass a status word to learn of them.
//   * The first call on each device resolves the array's device address
//     (cudaGetSymbolAddress, with that device current) and caches it; make that
//     first call before any stream capture.  The address belongs to the
//     context current at that call: after a device reset call pva_release (it
//     drops the cached address) before calling again.
#include <math.h>

#include <mutex>

#include "pva_internal.h"

using namespace pva;
using namespace pva::host;

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;   // whole array, per device
constexpr size_t kStatusBytes = 256;                 // internal status word
constexpr size_t kIntBytes = size_t(1) << 20;        // scheduler lists and counters
constexpr size_t kPartialBytes = kScratchBytes - kStatusBytes - kIntBytes;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a stand-in for the
// symbol; its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

struct DeviceScratch {
  unsigned char* base = nullptr;  // device address of g_scratch on this device
  int num_sms = 0;
};
std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

int device_scratch(int dev, DeviceScratch* out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(PVA_ERR_UNSUPPORTED, "device ordinal too large");
  DeviceScratch& d = g_dev[dev];
  if (!d.base) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(static scratch)");
    e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    d.base = static_cast<unsigned char*>(ptr);
  }
  *out = d;
  return PVA_OK;
}

}  // namespace

namespace pva {
namespace host {
void noalloc_forget_device(int dev) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (dev >= 0 && dev < kMaxDevices) g_dev[dev] = DeviceScratch{};
}
}  // namespace host
}  // namespace pva

extern "C" int pva_forward_noalloc(const void* q, const void* k, const void* v,
                                   const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv,
                                   void* out, int B, int num_heads, int kv_num_heads,
                                   int head_size, int v_head_size, float scale, int is_causal,
                                   float softcap, int dtype, uint32_t* device_status,
                                   void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  std::lock_guard<std::mutex> lock(g_mu);
  Plan plan;
  int rc = check_and_plan(q, k, v, cu_seqlens_q, cu_seqlens_kv, out, B, num_heads, kv_num_heads,
                          head_size, v_head_size, scale, softcap, dtype, &plan);
  if (rc != PVA_OK) return rc;
  if (plan.int_bytes > kIntBytes)
    return fail(PVA_ERR_UNSUPPORTED,
                "batch too large for the static scratch of pva_forward_noalloc "
                "(B * (4 + kv_num_heads) int32 words must stay within 1 MiB)");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceScratch ds;
  if ((rc = device_scratch(dev, &ds)) != PVA_OK) return rc;

  const int G = num_heads / kv_num_heads;
  int cap_units = 0;
  if (plan.decode) {
    const size_t per_unit = (size_t)(G * v_head_size + 2 * G) * sizeof(float);
    const size_t fit = kPartialBytes / per_unit;
    cap_units = (int)(fit < (size_t)plan.cap_units ? fit : (size_t)plan.cap_units);
  }
  uint32_t* status = device_status;
  if (!status) {
    status = reinterpret_cast<uint32_t*>(ds.base);
    e = cudaMemsetAsync(status, 0, sizeof(uint32_t), stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(status)");
  }
  plan.sched.num_sms = ds.num_sms;

  AttnParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.cu_q = cu_seqlens_q;
  p.cu_kv = cu_seqlens_kv;
  p.B = B;
  p.H = num_heads;
  p.Hkv = kv_num_heads;
  p.G = G;
  p.d = head_size;
  p.dv = v_head_size;
  p.scale = scale != 0.0f ? scale : 1.0f / sqrtf((float)head_size);
  p.softcap = fabsf(softcap);
  p.is_causal = is_causal ? 1 : 0;
  p.status = status;
  p.ws = reinterpret_cast<int32_t*>(ds.base + kStatusBytes);
  p.partials = reinterpret_cast<float*>(ds.base + kStatusBytes + kIntBytes);
  p.dec_cap_units = cap_units;

  CUtensorMap tq, tk, tv, to, dk, dvm;
  if (plan.tensor_core) {
    if ((rc = get_encoder()) != PVA_OK) return rc;
    const void* any = p.ws;  // stand-in address for empty (NULL) tensors
    const void* qa = q ? q : any;
    const void* ka = k ? k : any;
    const void* va = v ? v : any;
    const void* oa = out ? out : any;
    const int m = kTcRows / G, bn = tc_block_n(head_size, v_head_size);
    if ((rc = encode_map(&tq, qa, dtype, head_size, num_heads, 64, G, m, true)) != PVA_OK ||
        (rc = encode_map(&tk, ka, dtype, head_size, kv_num_heads, 64, 1, bn, true)) != PVA_OK ||
        (rc = encode_map(&tv, va, dtype, v_head_size, kv_num_heads, 64, 1, bn, true)) != PVA_OK ||
        (rc = encode_map(&to, oa, dtype, v_head_size, num_heads, 64, G, out_box_tokens(G),
                         true)) != PVA_OK)
      return rc;
    if (plan.decode) {
      const int tkeys = decode_tile_keys(head_size, v_head_size);
      if ((rc = encode_map(&dk, ka, dtype, head_size, kv_num_heads, head_size, 1, tkeys,
                           false)) != PVA_OK ||
          (rc = encode_map(&dvm, va, dtype, v_head_size, kv_num_heads, v_head_size, 1, tkeys,
                           false)) != PVA_OK)
        return rc;
    }
  }

  e = launch_scheduler(p, plan.sched, stream);
  if (e != cudaSuccess) return cuda_fail(e, "scheduler launch");
  if (!plan.tensor_core) {
    e = launch_prefill_f32(p, ds.num_sms, stream);
    return e == cudaSuccess ? PVA_OK : cuda_fail(e, "fp32 attention launch");
  }
  if (plan.decode) {  // decode first, as pva_forward orders them
    e = launch_decode(p, dtype, dk, dvm, ds.num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "split-KV decode launch");
  }
  e = tc_paired(head_size, v_head_size)
          ? launch_prefill_pair(p, dtype, tq, tk, tv, to, ds.num_sms, stream)
          : launch_prefill_tc(p, dtype, tq, tk, tv, to, ds.num_sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core prefill launch");
  return PVA_OK;
}
