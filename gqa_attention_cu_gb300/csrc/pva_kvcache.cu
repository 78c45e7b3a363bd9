// Front end of one GroupQueryAttention step against a fixed-capacity KV cache
// (group_query_attention.rs: `gqa_prepare_metadata`, `gqa_append_cache`,
// `gqa_rope_bnsh` and the fused single-token `gqa_fuse_decode_prep`).
//
//   pva_cache_meta_kernel  one CTA.  Per sequence: total = seqlens_k + 1,
//       past = total - k_seq (first appended cache row), query start =
//       total - q_seq; the step is rejected when any sequence breaks a bound
//       the page checks (total beyond int32, negative past or query start,
//       past or total beyond the capacity, a rotary position outside the
//       cos/sin tables), or when an earlier step on the stream was rejected
//       (the page's latch-first rule: a later in-range step must not append
//       after a row a rejected step skipped).  A rejected step latches
//       PVA_DEV_KV_CACHE and writes -1 lengths, so nothing is appended and the
//       scheduler gives the attention kernels no work; otherwise it writes the
//       offsets the scheduler reads (queries b * q_seq, cache planes b * cap,
//       key counts = totals).
//   pva_cache_prep_kernel  grid-stride over dimension pairs of the new rows:
//       appends K (rotated) and V at cache rows [past, past + k_seq) of every
//       (sequence, kv head) plane, and writes the rotated queries to scratch.
//       One launch replaces the page's separate append and rotary launches.
//
// The rotation of a pair (x0, x1) by (c, s) is computed in f32 with every
// product and sum rounded on its own, as the page's f32 kernel does
// (c*x0 - s*x1, s*x0 + c*x1), then rounded to the storage type.  Pairs are
// (2k, 2k+1) when interleaved, else (k, k + rot/2); dims past rot are copied.
#include "pva_device.cuh"

namespace pva {
namespace {

template <typename T>
__device__ __forceinline__ float to_f(T x) { return static_cast<float>(x); }
template <>
__device__ __forceinline__ float to_f<float>(float x) { return x; }

template <typename T>
__device__ __forceinline__ T from_f(float x);
template <>
__device__ __forceinline__ float from_f<float>(float x) { return x; }
template <>
__device__ __forceinline__ __half from_f<__half>(float x) { return __float2half_rn(x); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__device__ __forceinline__ float table(const void* t, int idx, int is_f16) {
  return is_f16 ? __half2float(static_cast<const __half*>(t)[idx])
                : static_cast<const float*>(t)[idx];
}

__global__ void __launch_bounds__(1024) pva_cache_meta_kernel(CacheStep c) {
  allow_next_grid();  // the append kernel may start its launch now
  wait_prior_grid();  // launched as a dependent of the work before it
  __shared__ uint32_t s_bad;
  if (threadIdx.x == 0) s_bad = (atomicOr(c.status, 0u) & PVA_DEV_KV_CACHE) ? 1u : 0u;
  __syncthreads();
  const int B = c.B;
  for (int b = threadIdx.x; b < B; b += blockDim.x) {
    const long long total = (long long)c.seqlens_k[b] + 1;
    const long long past = total - c.k_seq, first = total - c.q_seq;
    if (total > INT_MAX || past < 0 || first < 0 || past > c.cap || total > c.cap)
      atomicOr(&s_bad, 1u);
  }
  if (c.rot > 0) {
    // every rotated row's position must index the cos/sin tables; with no
    // position ids the rows of sequence b sit at first_b + s (queries) and
    // past_b + s (keys), equal here because k_seq is 0 or q_seq
    const long long n = (long long)B * c.q_seq;
    for (long long e = threadIdx.x; e < n; e += blockDim.x) {
      const int b = (int)(e / c.q_seq), s = (int)(e - (long long)b * c.q_seq);
      const long long pos = c.position_ids
                                ? c.position_ids[e]
                                : (long long)c.seqlens_k[b] + 1 - c.q_seq + s;
      if (pos < 0 || pos >= c.cache_rows) atomicOr(&s_bad, 1u);
    }
  }
  __syncthreads();
  const bool ok = s_bad == 0;
  for (int b = threadIdx.x; b <= B; b += blockDim.x) {
    c.cu_q[b] = b * c.q_seq;
    c.cu_kv[b] = b * c.cap;
    if (b < B) {
      const int total = c.seqlens_k[b] + 1;
      c.kv_len[b] = ok ? total : -1;
      c.past[b] = ok ? total - c.k_seq : -1;
      c.q_first[b] = ok ? total - c.q_seq : -1;
    }
  }
  if (threadIdx.x == 0 && !ok) atomicOr(c.status, PVA_DEV_KV_CACHE);
}

// Pair k of a head row: the two dims it covers and whether it is rotated.
__device__ __forceinline__ void pair_dims(int k, int rot, int interleaved, int& d0, int& d1,
                                          bool& rotated) {
  const int half = rot / 2;
  rotated = k < half;
  if (rotated) {
    d0 = interleaved ? 2 * k : k;
    d1 = interleaved ? 2 * k + 1 : k + half;
  } else {
    d0 = rot + 2 * (k - half);
    d1 = d0 + 1;
  }
}

template <typename T>
__global__ void __launch_bounds__(256) pva_cache_prep_kernel(CacheStep c) {
  // a programmatic dependent of the metadata kernel, whose starts it reads
  allow_next_grid();
  wait_prior_grid();
  const int hd = c.d / 2;  // pairs per head row
  const long long nq = c.rot > 0 ? (long long)c.B * c.q_seq * c.H * hd : 0;
  const long long nk = (long long)c.B * c.k_seq * c.Hkv * hd;
  const long long n = nq + 2 * nk;
  const T* q = static_cast<const T*>(c.q);
  const T* kn = static_cast<const T*>(c.k_new);
  const T* vn = static_cast<const T*>(c.v_new);
  T* kc = static_cast<T*>(c.k_cache);
  T* vc = static_cast<T*>(c.v_cache);
  T* qr = static_cast<T*>(c.q_rot);
  for (long long e = blockIdx.x * (long long)blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x) {
    long long x = e;
    const int region = x < nq ? 0 : (x < nq + nk ? 1 : 2);
    x -= region == 0 ? 0 : (region == 1 ? nq : nq + nk);
    const int heads = region == 0 ? c.H : c.Hkv;
    const int seq = region == 0 ? c.q_seq : c.k_seq;
    const int k = (int)(x % hd);
    x /= hd;
    const int h = (int)(x % heads);
    x /= heads;
    const int s = (int)(x % seq);
    const int b = (int)(x / seq);
    const int start = region == 0 ? c.q_first[b] : c.past[b];
    if (start < 0) continue;  // step rejected: nothing is written
    int d0, d1;
    bool rotated;
    pair_dims(k, c.rot, c.interleaved, d0, d1, rotated);
    const size_t src = ((size_t)(b * seq + s) * heads + h) * c.d;
    const T* in = region == 0 ? q : (region == 1 ? kn : vn);
    T* dst;
    if (region == 0)
      dst = qr + src;
    else
      dst = (region == 1 ? kc : vc) + ((size_t)(b * c.Hkv + h) * c.cap + start + s) * c.d;
    if (region == 2 || !rotated || c.rot == 0) {
      dst[d0] = in[src + d0];
      dst[d1] = in[src + d1];
      continue;
    }
    const long long pos = c.position_ids ? c.position_ids[(size_t)b * c.q_seq + s]
                                         : (long long)start + s;
    const int ti = (int)pos * (c.rot / 2) + k;
    const float co = table(c.cos_cache, ti, c.rot_f16), si = table(c.sin_cache, ti, c.rot_f16);
    const float x0 = to_f<T>(in[src + d0]), x1 = to_f<T>(in[src + d1]);
    dst[d0] = from_f<T>(__fsub_rn(__fmul_rn(co, x0), __fmul_rn(si, x1)));
    dst[d1] = from_f<T>(__fadd_rn(__fmul_rn(si, x0), __fmul_rn(co, x1)));
  }
}

}  // namespace

cudaError_t launch_cache_front(const CacheStep& c, cudaStream_t s) {
  cudaError_t e = launch_dependent(pva_cache_meta_kernel, dim3(1), dim3(1024), 0, s, c);
  if (e != cudaSuccess) return e;
  const long long hd = c.d / 2;
  const long long n = (c.rot > 0 ? (long long)c.B * c.q_seq * c.H * hd : 0) +
                      2LL * c.B * c.k_seq * c.Hkv * hd;
  if (n == 0) return cudaSuccess;
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long want = (n + 255) / 256, cap = (long long)(sms > 0 ? sms : 1) * 8;
  const int grid = (int)(want < cap ? want : cap);
  switch (c.dtype) {
    case PVA_F32:
      return launch_dependent(pva_cache_prep_kernel<float>, dim3(grid), dim3(256), 0, s, c);
    case PVA_F16:
      return launch_dependent(pva_cache_prep_kernel<__half>, dim3(grid), dim3(256), 0, s, c);
    default:
      return launch_dependent(pva_cache_prep_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, c);
  }
}

}  // namespace pva
