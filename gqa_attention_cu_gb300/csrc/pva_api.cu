// Host side of libpva: argument checks, per-(device, stream) workspaces,
// TMA tensor maps, and the launches of the scheduler and compute kernels.
//
// Argument rules follow the op's schema and the checks of its `execute`
// (packed_varlen_attention.rs: dtypes f32/f16/bf16, num_heads and
// kv_num_heads positive with kv_num_heads dividing num_heads, default scale
// 1/sqrt(head_size) computed in f32).  The offsets themselves are checked on
// the device (pva_scheduler.cu), so no call copies anything back to the host.
#include <cudaTypedefs.h>
#include <math.h>
#include <stdio.h>
#include <string.h>

#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <utility>

#include <climits>

#include "pva_internal.h"

using namespace pva;

namespace pva {
namespace host {

thread_local std::string g_last_error;

// Benchmark timing (pva_profile / pva_kernel_times): events around each launch.
struct Profile {
  bool enabled = false;
  bool have = false;
  bool decode = false;
  int dev = -1;
  cudaStream_t stream = nullptr;
  cudaEvent_t ev[4] = {nullptr, nullptr, nullptr, nullptr};
};
thread_local Profile g_prof;

void prof_mark(int i, cudaStream_t s) {
  if (!g_prof.enabled) return;
  if (!g_prof.ev[i]) cudaEventCreate(&g_prof.ev[i]);
  cudaEventRecord(g_prof.ev[i], s);
}

int fail(int code, const std::string& msg) {
  g_last_error = msg;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PVA_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct DeviceInfo {
  int num_sms = 0;
  bool ready = false;
};

struct Workspace {
  uint32_t* status = nullptr;  // sticky status word (never moves)
  void* buf = nullptr;         // int region + partials
  size_t bytes = 0;
};

std::mutex g_mu;
std::map<int, DeviceInfo> g_dev;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
// Resolved once per process; every entry point (whichever lock it holds)
// goes through get_encoder, so the lookup is guarded by its own once-flag.
std::atomic<PFN_cuTensorMapEncodeTiled_v12000> g_encode{nullptr};
std::once_flag g_encode_once;

int device_info(int dev, DeviceInfo* out) {
  auto& d = g_dev[dev];
  if (!d.ready) {
    cudaError_t e = cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute");
    d.ready = true;
  }
  *out = d;
  return PVA_OK;
}

int get_encoder() {
  std::call_once(g_encode_once, [] {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn)
      g_encode.store(reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn));
  });
  if (!g_encode.load())
    return fail(PVA_ERR_CUDA, "cuTensorMapEncodeTiled entry point not available");
  return PVA_OK;
}

// Rank-3 map over a packed [tokens, heads, dim] tensor of 16-bit elements.
// The token extent is set to INT32_MAX: the kernels never address a token
// outside [0, cu[B]) (tiles are shifted back at the end of the buffer and
// negative starts are zero-filled), so the extent is only a bound.
int encode_map(CUtensorMap* map, const void* base, int dtype, int dim, int heads, int box_dim,
               int box_heads, int box_tokens, bool swizzle128) {
  const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)INT32_MAX};
  const cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)dim * heads * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_dim, (cuuint32_t)box_heads, (cuuint32_t)box_tokens};
  const cuuint32_t estride[3] = {1, 1, 1};
  const auto encode = g_encode.load();
  CUresult r = encode(map, dtype == PVA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      3, const_cast<void*>(base), gdim, gstride, box, estride,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[160];
    snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (%d) dim=%d heads=%d box=%dx%dx%d",
             (int)r, dim, heads, box_dim, box_heads, box_tokens);
    return fail(PVA_ERR_CUDA, msg);
  }
  return PVA_OK;
}

// Rank-3 map over a BNSH cache [planes, rows, dim] (plane = sequence * Hkv +
// kv head, rows = the cache capacity): boxes of box_rows rows of one plane.
// Rows past the capacity read as zeros.
int encode_plane_map(CUtensorMap* map, const void* base, int dtype, int dim, int rows,
                     long long planes, int box_dim, int box_rows, bool swizzle128) {
  const cuuint64_t gdim[3] = {(cuuint64_t)dim, (cuuint64_t)rows, (cuuint64_t)planes};
  const cuuint64_t gstride[2] = {(cuuint64_t)dim * 2, (cuuint64_t)dim * rows * 2};
  const cuuint32_t box[3] = {(cuuint32_t)box_dim, (cuuint32_t)box_rows, 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  const auto encode = g_encode.load();
  CUresult r = encode(map, dtype == PVA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      3, const_cast<void*>(base), gdim, gstride, box, estride,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[160];
    snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (%d) dim=%d rows=%d planes=%lld",
             (int)r, dim, rows, planes);
    return fail(PVA_ERR_CUDA, msg);
  }
  return PVA_OK;
}

// Rank-4 map over padded slots [slots, rows, heads, dim] (the padded
// layout of the opset-24 nonpad_kv_seqlen input): boxes of box_rows rows of
// one kv head of one slot.  Rows outside [0, rows) of a slot read as zeros,
// so a tile never reaches into the next slot.
int encode_slot_map(CUtensorMap* map, const void* base, int dtype, int dim, int heads, int rows,
                    int slots, int box_dim, int box_rows, bool swizzle128) {
  const cuuint64_t gdim[4] = {(cuuint64_t)dim, (cuuint64_t)heads, (cuuint64_t)rows,
                              (cuuint64_t)slots};
  const cuuint64_t gstride[3] = {(cuuint64_t)dim * 2, (cuuint64_t)dim * heads * 2,
                                 (cuuint64_t)dim * heads * rows * 2};
  const cuuint32_t box[4] = {(cuuint32_t)box_dim, 1, (cuuint32_t)box_rows, 1};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  const auto encode = g_encode.load();
  CUresult r = encode(map, dtype == PVA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                             : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                      4, const_cast<void*>(base), gdim, gstride, box, estride,
                      CU_TENSOR_MAP_INTERLEAVE_NONE,
                      swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                      CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char msg[160];
    snprintf(msg, sizeof msg, "cuTensorMapEncodeTiled failed (%d) dim=%d heads=%d rows=%d slots=%d",
             (int)r, dim, heads, rows, slots);
    return fail(PVA_ERR_CUDA, msg);
  }
  return PVA_OK;
}

int check_and_plan(const void* q, const void* k, const void* v, const int32_t* cu_q,
                   const int32_t* cu_kv, void* out, int B, int H, int Hkv, int d, int dv,
                   float scale, float softcap, int dtype, Plan* plan) {
  // q/k/v/out may be NULL for empty tensors; the scheduler checks them
  // against the totals on the device.
  (void)q; (void)k; (void)v; (void)out;
  if (!cu_q || !cu_kv) return fail(PVA_ERR_INVALID_ARG, "null cu_seqlens pointer");
  if (B < 1) return fail(PVA_ERR_INVALID_ARG, "B must be >= 1");
  if (H <= 0 || Hkv <= 0 || H % Hkv != 0)
    return fail(PVA_ERR_INVALID_ARG,
                "num_heads must be a positive multiple of a positive kv_num_heads");
  if (dtype != PVA_F32 && dtype != PVA_F16 && dtype != PVA_BF16)
    return fail(PVA_ERR_INVALID_ARG, "dtype must be 0 (f32), 1 (f16) or 2 (bf16)");
  if (!isfinite(scale) || !isfinite(softcap))
    return fail(PVA_ERR_INVALID_ARG, "scale and softcap must be finite");
  if (d <= 0 || dv <= 0) return fail(PVA_ERR_INVALID_ARG, "head sizes must be positive");
  const int G = H / Hkv;
  if (dtype == PVA_F32) {
    if (d > 256 || dv > 256)
      return fail(PVA_ERR_UNSUPPORTED, "f32 path supports head sizes up to 256");
    plan->sched = SchedConfig{kF32TileTokens, H, kF32KeyTile, 0, 0, 0};
  } else {
    const bool shape_ok = (d == dv && (d == 64 || d == 96 || d == 128 || d == 192 || d == 256)) ||
                          (d == 192 && dv == 128);
    if (!shape_ok)
      return fail(PVA_ERR_UNSUPPORTED,
                  "f16/bf16 path supports (head_size, v_head_size) in {(64,64), (96,96), "
                  "(128,128), (192,192), (256,256), (192,128)}");
    if (G > kTcRows)
      return fail(PVA_ERR_UNSUPPORTED, "f16/bf16 path supports num_heads/kv_num_heads <= 128");
    const uintptr_t mis = (uintptr_t)q | (uintptr_t)k | (uintptr_t)v | (uintptr_t)out;
    if (mis & 15) return fail(PVA_ERR_INVALID_ARG, "q, k, v and out must be 16-byte aligned");
    plan->tensor_core = true;
    // The split-KV decode kernel covers every head-size pair of the
    // tensor-core path with G in {1, 2, 4, 8, 16}; other groupings take their
    // single-row sequences through the prefill kernel.  For d == dv in
    // {64, 128} with G <= 4 and d == dv == 256 with G <= 2 it reads K/V at
    // close to copy bandwidth and takes every single-row sequence; for the
    // other shapes (G = 8 and 16, d = 256 with G = 4, head sizes 96 and 192)
    // its arithmetic per K/V byte limits it, and the scheduler gives it
    // single-row sequences only when they are too few to keep every SM busy
    // in the prefill kernel (which does not split keys).
    plan->decode = G == 1 || G == 2 || G == 4 || G == 8 || G == 16;
    const bool tuned = d == dv && (((d == 64 || d == 128) && G <= 4) || (d == 256 && G <= 2));
    plan->sched = SchedConfig{(kTcRows / G) * tc_tiles_per_item(d, dv), Hkv, tc_block_n(d, dv),
                              plan->decode ? 1 : 0, 0, plan->decode && !tuned ? 1 : 0};
  }
  const WsLayout L{B, Hkv};
  plan->int_bytes = L.int_words() * 4;
  if (plan->decode) {
    long long cap = (long long)B * Hkv * kDecodeMaxSplits;
    if (cap > 16384) cap = 16384;
    plan->cap_units = (int)cap;
    plan->partial_bytes = (size_t)cap * (size_t)(G * dv + 2 * G) * sizeof(float);
  }
  return PVA_OK;
}

}  // namespace host
}  // namespace pva

using namespace pva::host;

namespace {

int get_workspace(int dev, cudaStream_t stream, size_t need, Workspace** out) {
  Workspace& w = g_ws[{dev, stream}];
  if (!w.status) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(stream, &cs);
    if (cs != cudaStreamCaptureStatusNone)
      return fail(PVA_ERR_INVALID_ARG,
                  "first call on a stream must not be captured (workspace allocation)");
    cudaError_t e = cudaMalloc(&w.status, 256);
    if (e != cudaSuccess) return fail(PVA_ERR_OOM, "status word allocation failed");
    e = cudaMemset(w.status, 0, 256);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset");
  }
  if (w.bytes < need) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaStreamIsCapturing(stream, &cs);
    if (cs != cudaStreamCaptureStatusNone)
      return fail(PVA_ERR_INVALID_ARG,
                  "workspace must grow but the stream is being captured; warm it up first");
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    if (w.buf) cudaFree(w.buf);
    w.buf = nullptr;
    w.bytes = 0;
    size_t sz = need < (1u << 20) ? (1u << 20) : need;
    e = cudaMalloc(&w.buf, sz);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return fail(PVA_ERR_OOM, "workspace allocation failed");
    }
    w.bytes = sz;
  }
  *out = &w;
  return PVA_OK;
}

int prepare(const void* q, const void* k, const void* v, const int32_t* cu_q,
            const int32_t* cu_kv, void* out, int B, int H, int Hkv, int d, int dv, float scale,
            int is_causal, float softcap, int dtype, cudaStream_t stream, Plan* plan,
            AttnParams* p, int* num_sms, size_t extra_int_words = 0) {
  int rc = check_and_plan(q, k, v, cu_q, cu_kv, out, B, H, Hkv, d, dv, scale, softcap, dtype,
                          plan);
  if (rc != PVA_OK) return rc;
  // room after the work lists for offsets the library builds itself
  plan->int_bytes += (extra_int_words * 4 + 255) / 256 * 256;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  DeviceInfo di;
  rc = device_info(dev, &di);
  if (rc != PVA_OK) return rc;
  *num_sms = di.num_sms;
  plan->sched.num_sms = di.num_sms;
  Workspace* w = nullptr;
  rc = get_workspace(dev, stream, plan->int_bytes + plan->partial_bytes, &w);
  if (rc != PVA_OK) return rc;

  AttnParams& P = *p;
  P.q = q;
  P.k = k;
  P.v = v;
  P.out = out;
  P.cu_q = cu_q;
  P.cu_kv = cu_kv;
  P.B = B;
  P.H = H;
  P.Hkv = Hkv;
  P.G = H / Hkv;
  P.d = d;
  P.dv = dv;
  // scale 0 selects the default 1/sqrt(head_size), computed in f32 as the
  // page does; softcap's sign does not matter (c * tanh(s / c) is even in c).
  P.scale = scale != 0.0f ? scale : 1.0f / sqrtf((float)d);
  P.softcap = fabsf(softcap);
  P.is_causal = is_causal ? 1 : 0;
  P.status = w->status;
  P.ws = static_cast<int32_t*>(w->buf);
  P.partials = reinterpret_cast<float*>(static_cast<uint8_t*>(w->buf) + plan->int_bytes);
  P.dec_cap_units = plan->cap_units;
  return PVA_OK;
}

// What one call computes, whichever entry point it came through.
struct Spec {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* cu_q;
  const int32_t* cu_kv;
  void* out;
  int B, H, Hkv, d, dv;
  float scale;
  int is_causal;
  float softcap;
  int window;
  int dtype;
  // padded form (pva_forward_padded): device int64 [B]; offsets built on the device
  const int64_t* nonpad = nullptr;
  int q_seq = 0, kv_seq = 0;
  // cache form (pva_gqa_kvcache): front end and K/V read from the cache planes
  const CacheStep* cache = nullptr;
};

int forward_impl(const Spec& s, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  std::lock_guard<std::mutex> lock(g_mu);
  Plan plan;
  AttnParams p{};
  int num_sms = 0;
  const int B = s.B;
  const size_t elt = s.dtype == PVA_F32 ? 4 : 2;
  // Library-built offsets sit after the work lists: [cu_q B+1][cu_kv B+1]
  // [kv_len B] (+ [past B][first query B] for the cache form), then, for a
  // rotary cache step, the rotated queries.
  size_t front_words = 0, qrot_bytes = 0;
  if (s.nonpad) front_words = 3 * (size_t)B + 2;
  if (s.cache) {
    front_words = ((5 * (size_t)B + 2 + 63) / 64) * 64;
    if (s.cache->rot > 0) qrot_bytes = (size_t)B * s.cache->q_seq * s.H * s.d * elt;
  }
  int rc = prepare(s.q, s.k, s.v, s.cu_q, s.cu_kv, s.out, B, s.H, s.Hkv, s.d, s.dv, s.scale,
                   s.is_causal, s.softcap, s.dtype, stream, &plan, &p, &num_sms,
                   front_words + (qrot_bytes + 3) / 4);
  if (rc != PVA_OK) return rc;
  p.window = s.window > 0 ? s.window : 0;
  int32_t* front = p.ws + WsLayout{B, s.Hkv}.int_words();
  CacheStep cs{};
  if (s.nonpad) {
    p.cu_q = front;
    p.cu_kv = front + B + 1;
    p.kv_len = front + 2 * B + 2;
    p.kv_slot = s.kv_seq;  // K/V through per-slot maps: padding is never loaded
  }
  if (s.cache) {
    cs = *s.cache;
    cs.cu_q = front;
    cs.cu_kv = front + B + 1;
    cs.kv_len = front + 2 * B + 2;
    cs.past = front + 3 * B + 2;
    cs.q_first = front + 4 * B + 2;
    cs.status = p.status;
    cs.q_rot = qrot_bytes ? static_cast<void*>(front + front_words) : nullptr;
    p.cu_q = cs.cu_q;
    p.cu_kv = cs.cu_kv;
    p.kv_len = cs.kv_len;
    p.kv_cap = cs.cap;
    if (cs.q_rot) p.q = cs.q_rot;
  }

  CUtensorMap tq, tk, tv, to, dk, dvm;
  if (plan.tensor_core) {
    if ((rc = get_encoder()) != PVA_OK) return rc;
    // An empty tensor may come as NULL; its map is never used (the device
    // check empties the work lists), but the encoder wants a real address.
    const void* any = p.ws;
    const void* q = p.q ? p.q : any;
    const void* k = s.k ? s.k : any;
    const void* v = s.v ? s.v : any;
    void* o = s.out ? s.out : p.ws;
    const int G = p.G, m = kTcRows / G, bn = tc_block_n(s.d, s.dv);
    if ((rc = encode_map(&tq, q, s.dtype, s.d, s.H, 64, G, m, true)) != PVA_OK ||
        (rc = encode_map(&to, o, s.dtype, s.dv, s.H, 64, G, out_box_tokens(G), true)) !=
            PVA_OK)
      return rc;
    if (s.cache) {
      const long long planes = (long long)B * s.Hkv;
      if ((rc = encode_plane_map(&tk, k, s.dtype, s.d, cs.cap, planes, 64, bn, true)) !=
              PVA_OK ||
          (rc = encode_plane_map(&tv, v, s.dtype, s.dv, cs.cap, planes, 64, bn, true)) !=
              PVA_OK)
        return rc;
      if (plan.decode) {
        const int tkeys = decode_tile_keys(s.d, s.dv);
        if ((rc = encode_plane_map(&dk, k, s.dtype, s.d, cs.cap, planes, s.d, tkeys,
                                   false)) != PVA_OK ||
            (rc = encode_plane_map(&dvm, v, s.dtype, s.dv, cs.cap, planes, s.dv, tkeys,
                                   false)) != PVA_OK)
          return rc;
      }
    } else if (p.kv_slot) {
      if ((rc = encode_slot_map(&tk, k, s.dtype, s.d, s.Hkv, p.kv_slot, B, 64, bn, true)) !=
              PVA_OK ||
          (rc = encode_slot_map(&tv, v, s.dtype, s.dv, s.Hkv, p.kv_slot, B, 64, bn, true)) !=
              PVA_OK)
        return rc;
      if (plan.decode) {
        const int tkeys = decode_tile_keys(s.d, s.dv);
        if ((rc = encode_slot_map(&dk, k, s.dtype, s.d, s.Hkv, p.kv_slot, B, s.d, tkeys,
                                  false)) != PVA_OK ||
            (rc = encode_slot_map(&dvm, v, s.dtype, s.dv, s.Hkv, p.kv_slot, B, s.dv, tkeys,
                                  false)) != PVA_OK)
          return rc;
      }
    } else {
      if ((rc = encode_map(&tk, k, s.dtype, s.d, s.Hkv, 64, 1, bn, true)) != PVA_OK ||
          (rc = encode_map(&tv, v, s.dtype, s.dv, s.Hkv, 64, 1, bn, true)) != PVA_OK)
        return rc;
      if (plan.decode) {
        const int tkeys = decode_tile_keys(s.d, s.dv);
        if ((rc = encode_map(&dk, k, s.dtype, s.d, s.Hkv, s.d, 1, tkeys, false)) != PVA_OK ||
            (rc = encode_map(&dvm, v, s.dtype, s.dv, s.Hkv, s.dv, 1, tkeys, false)) != PVA_OK)
          return rc;
      }
    }
  }

  if (g_prof.enabled) {
    g_prof.have = true;
    g_prof.decode = plan.decode;
    g_prof.stream = stream;
    cudaGetDevice(&g_prof.dev);
  }
  prof_mark(0, stream);
  cudaError_t e = cudaSuccess;
  if (s.nonpad) {
    e = launch_padded_front(s.nonpad, B, s.q_seq, s.kv_seq, front, front + B + 1,
                            front + 2 * B + 2, stream);
    if (e != cudaSuccess) return cuda_fail(e, "padded front-end launch");
  }
  if (s.cache) {
    e = launch_cache_front(cs, stream);
    if (e != cudaSuccess) return cuda_fail(e, "kv-cache front-end launch");
  }
  e = launch_scheduler(p, plan.sched, stream);
  if (e != cudaSuccess) return cuda_fail(e, "scheduler launch");
  prof_mark(1, stream);
  if (!plan.tensor_core) {
    e = launch_prefill_f32(p, num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "fp32 attention launch");
    prof_mark(2, stream);
    return PVA_OK;
  }
  // The decode kernel goes first: a batch without single-row sequences gives
  // it no units, and it then exits while the scheduler's successor chain is
  // still starting, instead of adding a launch after the prefill kernel.
  if (plan.decode) {
    e = launch_decode(p, s.dtype, dk, dvm, num_sms, stream);
    if (e != cudaSuccess) return cuda_fail(e, "split-KV decode launch");
    prof_mark(2, stream);
  }
  e = tc_paired(s.d, s.dv) ? launch_prefill_pair(p, s.dtype, tq, tk, tv, to, num_sms, stream)
                           : launch_prefill_tc(p, s.dtype, tq, tk, tv, to, num_sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "tensor-core prefill launch");
  prof_mark(plan.decode ? 3 : 2, stream);
  return PVA_OK;
}

// ---- host-buffer entry point (pva_forward_from_host) -------------------------
constexpr int kMaxChunks = 16;

struct ChunkBounds {
  int n;                   // chunks
  int b0[kMaxChunks + 1];  // first sequence of each chunk; b0[n] = B
};

// Offsets of each chunk rebased to its first sequence: chunk c's sequences
// [b0[c], b0[c+1]) get cu - cu[b0[c]], written from index b0[c] + c on (one
// block per chunk).
__global__ void pva_rebase_kernel(const int32_t* cu_q, const int32_t* cu_kv, ChunkBounds cb,
                                  int32_t* out_q, int32_t* out_kv) {
  const int c = blockIdx.x;
  if (c >= cb.n) return;
  const int b0 = cb.b0[c], b1 = cb.b0[c + 1];
  const int q0 = cu_q[b0], k0 = cu_kv[b0];
  for (int i = threadIdx.x; i <= b1 - b0; i += blockDim.x) {
    out_q[b0 + c + i] = cu_q[b0 + i] - q0;
    out_kv[b0 + c + i] = cu_kv[b0 + i] - k0;
  }
}

// Copy streams and events of the host-buffer entry point, one set per device.
struct HostPipe {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t in_ev[kMaxChunks] = {}, comp_ev[kMaxChunks] = {};
};
std::mutex g_pipe_mu;
std::map<int, HostPipe> g_pipe;

int get_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    cudaError_t e;
    if (!hp.in && (e = cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking)) != cudaSuccess)
      return cuda_fail(e, "cudaStreamCreateWithFlags");
    if (!hp.out && (e = cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking)) != cudaSuccess)
      return cuda_fail(e, "cudaStreamCreateWithFlags");
    cudaEvent_t* evs[2 + 2 * kMaxChunks];
    int ne = 0;
    evs[ne++] = &hp.start;
    evs[ne++] = &hp.done;
    for (int c = 0; c < kMaxChunks; ++c) {
      evs[ne++] = &hp.in_ev[c];
      evs[ne++] = &hp.comp_ev[c];
    }
    for (int i = 0; i < ne; ++i)
      if (!*evs[i] && (e = cudaEventCreateWithFlags(evs[i], cudaEventDisableTiming)) != cudaSuccess)
        return cuda_fail(e, "cudaEventCreateWithFlags");
    hp.ready = true;
  }
  *out = &hp;
  return PVA_OK;
}

}  // namespace

extern "C" {

int pva_forward(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                const int32_t* cu_seqlens_kv, void* out, int B, int num_heads, int kv_num_heads,
                int head_size, int v_head_size, float scale, int is_causal, float softcap,
                int dtype, void* stream) {
  const Spec s{q, k, v, cu_seqlens_q, cu_seqlens_kv, out, B, num_heads, kv_num_heads,
               head_size, v_head_size, scale, is_causal, softcap, 0, dtype};
  return forward_impl(s, stream);
}

int pva_forward_local(const void* q, const void* k, const void* v, const int32_t* cu_seqlens_q,
                      const int32_t* cu_seqlens_kv, void* out, int B, int num_heads,
                      int kv_num_heads, int head_size, int v_head_size, float scale,
                      int is_causal, float softcap, int local_window, int dtype, void* stream) {
  const Spec s{q, k, v, cu_seqlens_q, cu_seqlens_kv, out, B, num_heads, kv_num_heads,
               head_size, v_head_size, scale, is_causal, softcap, local_window, dtype};
  return forward_impl(s, stream);
}

int pva_forward_padded(const void* q, const void* k, const void* v,
                       const int64_t* nonpad_kv_seqlen, void* out, int B, int q_seq, int kv_seq,
                       int num_heads, int kv_num_heads, int head_size, int v_head_size,
                       float scale, int is_causal, float softcap, int dtype, void* stream) {
  if (!nonpad_kv_seqlen) return fail(PVA_ERR_INVALID_ARG, "null nonpad_kv_seqlen pointer");
  if (B < 1) return fail(PVA_ERR_INVALID_ARG, "B must be >= 1");
  if (q_seq < 0 || kv_seq < 0)
    return fail(PVA_ERR_INVALID_ARG, "q_seq and kv_seq must be non-negative");
  if ((long long)B * q_seq > INT_MAX || (long long)B * kv_seq > INT_MAX)
    return fail(PVA_ERR_INVALID_ARG, "B * q_seq and B * kv_seq must fit in int32");
  // The offsets are built on the device; the nonpad pointer stands in for them
  // in the host checks (which only test that they are non-null).
  const int32_t* stand_in = reinterpret_cast<const int32_t*>(nonpad_kv_seqlen);
  Spec s{q, k, v, stand_in, stand_in, out, B, num_heads, kv_num_heads, head_size,
         v_head_size, scale, is_causal, softcap, 0, dtype};
  s.nonpad = nonpad_kv_seqlen;
  s.q_seq = q_seq;
  s.kv_seq = kv_seq;
  return forward_impl(s, stream);
}

int pva_gqa_kvcache(const void* q, const void* k_new, const void* v_new, void* k_cache,
                    void* v_cache, const int32_t* seqlens_k, const void* cos_cache,
                    const void* sin_cache, const int64_t* position_ids, void* out, int B,
                    int q_seq, int k_seq, int capacity, int num_heads, int kv_num_heads,
                    int head_size, int rotary_dim, int cache_rows, int rotary_interleaved,
                    int rotary_dtype, float scale, float softcap, int local_window, int dtype,
                    void* stream) {
  if (!q || !k_cache || !v_cache || !out || !seqlens_k)
    return fail(PVA_ERR_INVALID_ARG, "null q, cache, out or seqlens_k pointer");
  if (B < 1 || q_seq < 1 || k_seq < 0 || capacity < 1)
    return fail(PVA_ERR_INVALID_ARG, "need B >= 1, q_seq >= 1, k_seq >= 0, capacity >= 1");
  if (k_seq > 0 && (!k_new || !v_new))
    return fail(PVA_ERR_INVALID_ARG, "null k_new or v_new with k_seq > 0");
  if ((long long)(B + 1) * capacity > INT_MAX - 65536 || (long long)B * q_seq > INT_MAX ||
      (long long)B * k_seq > INT_MAX)
    return fail(PVA_ERR_INVALID_ARG, "cache or token extents do not fit in int32");
  if (head_size % 2 != 0) return fail(PVA_ERR_UNSUPPORTED, "head_size must be even");
  if (rotary_dim != 0) {
    if (rotary_dim < 2 || rotary_dim % 2 != 0 || rotary_dim > head_size)
      return fail(PVA_ERR_INVALID_ARG, "rotary_dim must be even with 2 <= rotary_dim <= head_size");
    if (!cos_cache || !sin_cache || cache_rows < 1)
      return fail(PVA_ERR_INVALID_ARG, "rotary embedding needs cos/sin tables with rows >= 1");
    if ((long long)cache_rows * (rotary_dim / 2) > INT_MAX)
      return fail(PVA_ERR_INVALID_ARG, "cos/sin tables too large");
    if (k_seq != 0 && k_seq != q_seq)
      return fail(PVA_ERR_INVALID_ARG, "rotary embedding needs k_seq == q_seq (or k_seq == 0)");
    if (rotary_dtype != PVA_F32 && !(rotary_dtype == PVA_F16 && dtype != PVA_F32))
      return fail(PVA_ERR_INVALID_ARG,
                  "cos/sin tables must be f32, or f16 with f16/bf16 queries");
  }
  CacheStep c{};
  c.q = q;
  c.k_new = k_new;
  c.v_new = v_new;
  c.k_cache = k_cache;
  c.v_cache = v_cache;
  c.seqlens_k = seqlens_k;
  c.cos_cache = cos_cache;
  c.sin_cache = sin_cache;
  c.position_ids = position_ids;
  c.B = B;
  c.q_seq = q_seq;
  c.k_seq = k_seq;
  c.cap = capacity;
  c.H = num_heads;
  c.Hkv = kv_num_heads;
  c.d = head_size;
  c.rot = rotary_dim;
  c.cache_rows = cache_rows;
  c.interleaved = rotary_interleaved ? 1 : 0;
  c.rot_f16 = rotary_dtype == PVA_F16 ? 1 : 0;
  c.dtype = dtype;
  // The attention reads the cache planes; seqlens_k stands in for the offsets
  // in the host checks (which only test that they are non-null).
  Spec s{q, k_cache, v_cache, seqlens_k, seqlens_k, out, B, num_heads, kv_num_heads,
         head_size, head_size, scale, 1, softcap, local_window, dtype};
  s.cache = &c;
  return forward_impl(s, stream);
}

int pva_get_status(void* stream_, uint32_t* device_flags) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!device_flags) return fail(PVA_ERR_INVALID_ARG, "device_flags is null");
  *device_flags = 0;
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  auto it = g_ws.find({dev, stream});
  if (it == g_ws.end() || !it->second.status) return PVA_OK;
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  uint32_t v = 0;
  e = cudaMemcpy(&v, it->second.status, sizeof v, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy status");
  e = cudaMemset(it->second.status, 0, sizeof v);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemset status");
  *device_flags = v;
  return PVA_OK;
}

int pva_schedule(const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_kv, int B, int num_heads,
                 int kv_num_heads, int head_size, int v_head_size, int is_causal, int dtype,
                 int32_t* host_out, size_t capacity, void* stream_) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  if (!host_out) return fail(PVA_ERR_INVALID_ARG, "host_out is null");
  if (B >= 1 && capacity < (size_t)8 + 4 * (size_t)B + 2)
    return fail(PVA_ERR_INVALID_ARG, "host_out capacity too small");
  std::lock_guard<std::mutex> lock(g_mu);
  Plan plan;
  AttnParams p{};
  int num_sms = 0;
  // q/k/v/out are not touched by the scheduler; aligned placeholders satisfy
  // the pointer checks.
  const void* dummy = reinterpret_cast<const void*>(uintptr_t(256));
  int rc = prepare(dummy, dummy, dummy, cu_seqlens_q, cu_seqlens_kv, const_cast<void*>(dummy), B,
                   num_heads, kv_num_heads, head_size, v_head_size, 1.0f, is_causal, 0.0f, dtype,
                   stream, &plan, &p, &num_sms);
  if (rc != PVA_OK) return rc;
  cudaError_t e = launch_scheduler(p, plan.sched, stream);
  if (e != cudaSuccess) return cuda_fail(e, "scheduler launch");
  const size_t words = 8 + 4 * (size_t)B + 2;
  e = cudaMemcpyAsync(host_out, p.ws, words * 4, cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpyAsync");
  e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  return PVA_OK;
}

int pva_selftest_wait(uint32_t limit_us, void* stream_, uint32_t* device_flags) {
  if (!device_flags) return fail(PVA_ERR_INVALID_ARG, "device_flags is null");
  if (limit_us < 1 || limit_us > 1000000)
    return fail(PVA_ERR_INVALID_ARG, "limit_us must be in 1..1000000");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  uint32_t* dev = nullptr;
  cudaError_t e = cudaMalloc(&dev, 16);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMalloc");
  uint32_t host[2] = {0, 0};
  e = cudaMemsetAsync(dev, 0, 16, stream);
  if (e == cudaSuccess)
    e = launch_wait_selftest(dev, (uint64_t)limit_us * 1000ull, reinterpret_cast<int*>(dev + 1),
                             stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(host, dev, 8, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  cudaFree(dev);
  if (e != cudaSuccess) return cuda_fail(e, "wait self-test");
  if (host[1] == 0) return fail(PVA_ERR_CUDA, "wait self-test kernel did not finish");
  *device_flags = host[0];
  return PVA_OK;
}

int pva_profile(int enable) {
  g_prof.enabled = enable != 0;
  g_prof.have = false;
  return PVA_OK;
}

int pva_kernel_times(float* ms, int capacity) {
  if (!ms || capacity < 3) return fail(PVA_ERR_INVALID_ARG, "need room for 3 durations");
  if (!g_prof.have) return fail(PVA_ERR_INVALID_ARG, "no profiled call yet");
  cudaError_t e = cudaStreamSynchronize(g_prof.stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
  ms[0] = ms[1] = ms[2] = -1.0f;
  cudaEventElapsedTime(&ms[0], g_prof.ev[0], g_prof.ev[1]);
  if (g_prof.decode) {
    // launch order: scheduler, decode, prefill
    cudaEventElapsedTime(&ms[2], g_prof.ev[1], g_prof.ev[2]);
    cudaEventElapsedTime(&ms[1], g_prof.ev[2], g_prof.ev[3]);
  } else {
    cudaEventElapsedTime(&ms[1], g_prof.ev[1], g_prof.ev[2]);
  }
  return PVA_OK;
}

const char* pva_status_string(int code) {
  switch (code) {
    case PVA_OK: return "ok";
    case PVA_ERR_INVALID_ARG: return "invalid argument";
    case PVA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PVA_ERR_CUDA: return "CUDA error";
    case PVA_ERR_OOM: return "out of device memory";
    default: return "unknown status";
  }
}

const char* pva_last_error(void) { return g_last_error.c_str(); }

void pva_release(void) {
  std::lock_guard<std::mutex> pipe_lock(g_pipe_mu);
  std::lock_guard<std::mutex> lock(g_mu);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return;
  cudaDeviceSynchronize();
  noalloc_forget_device(dev);
  auto hp = g_pipe.find(dev);
  if (hp != g_pipe.end()) {
    HostPipe& h = hp->second;
    if (h.in) cudaStreamDestroy(h.in);
    if (h.out) cudaStreamDestroy(h.out);
    cudaEvent_t evs[2 + 2 * kMaxChunks] = {h.start, h.done};
    for (int c = 0; c < kMaxChunks; ++c) {
      evs[2 + 2 * c] = h.in_ev[c];
      evs[3 + 2 * c] = h.comp_ev[c];
    }
    for (cudaEvent_t e : evs)
      if (e) cudaEventDestroy(e);
    g_pipe.erase(hp);
  }
  for (auto it = g_ws.begin(); it != g_ws.end();) {
    if (it->first.first == dev) {
      if (it->second.buf) cudaFree(it->second.buf);
      if (it->second.status) cudaFree(it->second.status);
      it = g_ws.erase(it);
    } else {
      ++it;
    }
  }
}

int pva_forward_from_host(const void* q_host, const void* k_host, const void* v_host,
                          const int32_t* cu_seqlens_q_host, const int32_t* cu_seqlens_kv_host,
                          void* out_host, void* q_dev, void* k_dev, void* v_dev, void* out_dev,
                          int32_t* cu_dev, int B, int num_heads, int kv_num_heads, int head_size,
                          int v_head_size, float scale, int is_causal, float softcap, int dtype,
                          int chunks, void* stream_) {
  if (B < 1 || !cu_seqlens_q_host || !cu_seqlens_kv_host || !cu_dev)
    return fail(PVA_ERR_INVALID_ARG, "B >= 1 and the offset arrays are required");
  if (num_heads <= 0 || kv_num_heads <= 0 || head_size <= 0 || v_head_size <= 0)
    return fail(PVA_ERR_INVALID_ARG, "head counts and sizes must be positive");
  if (dtype != PVA_F32 && dtype != PVA_F16 && dtype != PVA_BF16)
    return fail(PVA_ERR_INVALID_ARG, "dtype must be PVA_F32, PVA_F16 or PVA_BF16");
  // The copies are sized from the offsets, so they are checked here, on the
  // host, before anything is enqueued.
  if (cu_seqlens_q_host[0] != 0 || cu_seqlens_kv_host[0] != 0)
    return fail(PVA_ERR_INVALID_ARG, "cu_seqlens must start at 0");
  for (int b = 0; b < B; ++b)
    if (cu_seqlens_q_host[b + 1] < cu_seqlens_q_host[b] ||
        cu_seqlens_kv_host[b + 1] < cu_seqlens_kv_host[b])
      return fail(PVA_ERR_INVALID_ARG, "cu_seqlens must be non-decreasing");
  const long long tq = cu_seqlens_q_host[B], tk = cu_seqlens_kv_host[B];
  if ((tq > 0 && (!q_host || !q_dev || !out_host || !out_dev)) ||
      (tk > 0 && (!k_host || !v_host || !k_dev || !v_dev)))
    return fail(PVA_ERR_INVALID_ARG, "null buffer with a non-empty extent");
  const size_t esz = dtype == PVA_F32 ? 4 : 2;
  const size_t rq = (size_t)num_heads * head_size * esz, ro = (size_t)num_heads * v_head_size * esz;
  const size_t rk = (size_t)kv_num_heads * head_size * esz;
  const size_t rv = (size_t)kv_num_heads * v_head_size * esz;
  // Chunks: runs of whole sequences moving about equal bytes.
  int n = chunks <= 0 ? 8 : chunks;
  n = n < kMaxChunks ? n : kMaxChunks;
  n = n < B ? n : B;
  ChunkBounds cb{};
  {
    const double total = (double)tq * (rq + ro) + (double)tk * (rk + rv);
    double acc = 0.0;
    int c = 0;
    for (int b = 0; b + 1 < B && c + 1 < n; ++b) {
      acc += (double)(cu_seqlens_q_host[b + 1] - cu_seqlens_q_host[b]) * (rq + ro) +
             (double)(cu_seqlens_kv_host[b + 1] - cu_seqlens_kv_host[b]) * (rk + rv);
      if (acc >= total * (c + 1) / n) cb.b0[++c] = b + 1;
    }
    cb.n = c + 1;
    cb.b0[cb.n] = B;
  }
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  cudaStream_t s = static_cast<cudaStream_t>(stream_);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  HostPipe* hp = nullptr;
  int rc = get_pipe(dev, &hp);
  if (rc != PVA_OK) return rc;
  auto ck = [&](cudaError_t err, const char* what) { return err == cudaSuccess ? PVA_OK : cuda_fail(err, what); };
  // The copies start after the work already on `stream`, which may still read
  // the device buffers.
  if ((rc = ck(cudaEventRecord(hp->start, s), "cudaEventRecord")) != PVA_OK ||
      (rc = ck(cudaStreamWaitEvent(hp->in, hp->start, 0), "cudaStreamWaitEvent")) != PVA_OK)
    return rc;
  int32_t* cu_q_d = cu_dev;
  int32_t* cu_kv_d = cu_dev + (B + 1);
  int32_t* rq_d = cu_dev + 2 * (B + 1);
  int32_t* rkv_d = rq_d + (B + kMaxChunks);
  if ((rc = ck(cudaMemcpyAsync(cu_q_d, cu_seqlens_q_host, (B + 1) * sizeof(int32_t),
                               cudaMemcpyHostToDevice, hp->in), "cudaMemcpyAsync")) != PVA_OK ||
      (rc = ck(cudaMemcpyAsync(cu_kv_d, cu_seqlens_kv_host, (B + 1) * sizeof(int32_t),
                               cudaMemcpyHostToDevice, hp->in), "cudaMemcpyAsync")) != PVA_OK)
    return rc;
  pva_rebase_kernel<<<cb.n, 128, 0, hp->in>>>(cu_q_d, cu_kv_d, cb, rq_d, rkv_d);
  if ((rc = ck(cudaGetLastError(), "pva_rebase_kernel launch")) != PVA_OK) return rc;
  auto at = [](const void* base, size_t off) {
    return const_cast<char*>(static_cast<const char*>(base)) + off;
  };
  for (int c = 0; c < cb.n; ++c) {
    const int b0 = cb.b0[c], b1 = cb.b0[c + 1];
    const size_t q0 = cu_seqlens_q_host[b0], q1 = cu_seqlens_q_host[b1];
    const size_t k0 = cu_seqlens_kv_host[b0], k1 = cu_seqlens_kv_host[b1];
    // this chunk's rows in, on the copy-in stream
    if (q1 > q0 && (rc = ck(cudaMemcpyAsync(at(q_dev, q0 * rq), at(q_host, q0 * rq), (q1 - q0) * rq,
                                            cudaMemcpyHostToDevice, hp->in), "cudaMemcpyAsync")) != PVA_OK)
      return rc;
    if (k1 > k0 &&
        ((rc = ck(cudaMemcpyAsync(at(k_dev, k0 * rk), at(k_host, k0 * rk), (k1 - k0) * rk,
                                  cudaMemcpyHostToDevice, hp->in), "cudaMemcpyAsync")) != PVA_OK ||
         (rc = ck(cudaMemcpyAsync(at(v_dev, k0 * rv), at(v_host, k0 * rv), (k1 - k0) * rv,
                                  cudaMemcpyHostToDevice, hp->in), "cudaMemcpyAsync")) != PVA_OK))
      return rc;
    if ((rc = ck(cudaEventRecord(hp->in_ev[c], hp->in), "cudaEventRecord")) != PVA_OK ||
        (rc = ck(cudaStreamWaitEvent(s, hp->in_ev[c], 0), "cudaStreamWaitEvent")) != PVA_OK)
      return rc;
    // its attention on `stream`
    if (q1 > q0 &&
        (rc = pva_forward(at(q_dev, q0 * rq), k1 > k0 ? at(k_dev, k0 * rk) : k_dev,
                          k1 > k0 ? at(v_dev, k0 * rv) : v_dev, rq_d + b0 + c, rkv_d + b0 + c,
                          at(out_dev, q0 * ro), b1 - b0, num_heads, kv_num_heads, head_size,
                          v_head_size, scale, is_causal, softcap, dtype, s)) != PVA_OK)
      return rc;
    // and its output rows back, on the copy-out stream
    if ((rc = ck(cudaEventRecord(hp->comp_ev[c], s), "cudaEventRecord")) != PVA_OK ||
        (rc = ck(cudaStreamWaitEvent(hp->out, hp->comp_ev[c], 0), "cudaStreamWaitEvent")) != PVA_OK)
      return rc;
    if (q1 > q0 && (rc = ck(cudaMemcpyAsync(at(out_host, q0 * ro), at(out_dev, q0 * ro),
                                            (q1 - q0) * ro, cudaMemcpyDeviceToHost, hp->out),
                            "cudaMemcpyAsync")) != PVA_OK)
      return rc;
  }
  // `stream` completes after the last output copy.
  if ((rc = ck(cudaEventRecord(hp->done, hp->out), "cudaEventRecord")) != PVA_OK ||
      (rc = ck(cudaStreamWaitEvent(s, hp->done, 0), "cudaStreamWaitEvent")) != PVA_OK)
    return rc;
  return PVA_OK;
}

int pva_version(void) { return (0 << 16) | (1 << 8) | 0; }

}  // extern "C"
