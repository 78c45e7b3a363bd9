// fp32 path (dtype 0): tiled online-softmax attention on the CUDA cores in
// exact fp32 (no TF32), for any head sizes 1..256.
//
// Same arithmetic as the page's kernel stages (packed_varlen_attention.rs,
// stages 1-5: scale * q.k, softcap before the mask, tail-aligned causal
// frontier, max-subtracted exponentials, zero rows when nothing is visible,
// weighted sum of V) but streamed over key tiles with a running maximum,
// so nothing of size L_kv is stored.
//
// Work item: (sequence, 16-token query tile, query head), taken from the
// scheduler's longest-first list by a persistent grid.  A CTA of 4 warps
// stages the tile's queries and 32-key K/V tiles in shared memory; each warp
// owns 4 query rows; lane j scores key j of the tile, lane c accumulates
// output channels c, c+32, ...
#include "pva_device.cuh"
#include "pva_items.cuh"

namespace pva {
namespace {

constexpr int kWarps = 4;
constexpr int kRowsPerWarp = kF32TileTokens / kWarps;  // 4
constexpr int kMaxDim = 256;
constexpr int kChan = kMaxDim / 32;                     // output channels per lane

__global__ void __launch_bounds__(kWarps * 32) pva_prefill_f32_kernel(AttnParams p) {
  extern __shared__ float smem[];
  const int d = p.d, dv = p.dv, kstride = d + 1;
  float* sq = smem;                              // [16][d]
  float* sk = sq + kF32TileTokens * d;           // [32][d+1]
  float* sv = sk + kF32KeyTile * kstride;        // [32][dv]

  wait_prior_grid();  // the scheduler's work lists are complete from here on
  const SchedHeader h = *reinterpret_cast<const SchedHeader*>(p.ws + kWsHeader);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const float* Q = static_cast<const float*>(p.q);
  const float* K = static_cast<const float*>(p.k);
  const float* V = static_cast<const float*>(p.v);
  float* O = static_cast<float*>(p.out);
  const float NEG_INF = __int_as_float(0xff800000);

  for (int it = blockIdx.x; it < h.n_items; it += gridDim.x) {
    const PrefillItem item = decode_prefill_item(p, h, it);
    const int hh = item.unit;                 // query head
    const int g = hh / p.G;                   // shared kv head
    const int row0 = item.t * kF32TileTokens;  // first local query row
    const int nrows = min(kF32TileTokens, item.lq - row0);
    const int off = item.lkv - item.lq;
    const int hi = item_key_extent(item, kF32TileTokens, p.is_causal);
    const int kb = item_key_begin(item, kF32TileTokens, p.window) / kF32KeyTile * kF32KeyTile;

    __syncthreads();  // previous item done with shared memory
    for (int e = threadIdx.x; e < kF32TileTokens * d; e += blockDim.x) {
      const int r = e / d, c = e - r * d;
      sq[e] = r < nrows ? Q[((size_t)(item.q_start + row0 + r) * p.H + hh) * d + c] : 0.0f;
    }

    float m[kRowsPerWarp], l[kRowsPerWarp], acc[kRowsPerWarp][kChan];
#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      m[r] = NEG_INF;
      l[r] = 0.0f;
#pragma unroll
      for (int u = 0; u < kChan; ++u) acc[r][u] = 0.0f;
    }

    for (int k0 = kb; k0 < hi; k0 += kF32KeyTile) {
      const int nk = min(kF32KeyTile, hi - k0);
      __syncthreads();  // previous key tile consumed
      for (int e = threadIdx.x; e < kF32KeyTile * d; e += blockDim.x) {
        const int j = e / d, c = e - j * d;
        sk[j * kstride + c] =
            j < nk ? K[kv_row(p, item.b, item.kv_start, g, k0 + j) * d + c] : 0.0f;
      }
      for (int e = threadIdx.x; e < kF32KeyTile * dv; e += blockDim.x) {
        const int j = e / dv, c = e - j * dv;
        sv[e] = j < nk ? V[kv_row(p, item.b, item.kv_start, g, k0 + j) * dv + c] : 0.0f;
      }
      __syncthreads();

#pragma unroll
      for (int r = 0; r < kRowsPerWarp; ++r) {
        const int lr = warp * kRowsPerWarp + r;  // row within the tile
        if (lr >= nrows) continue;               // warp-uniform
        const int i = row0 + lr;                 // local query position
        const int key = k0 + lane;
        bool visible = lane < nk;
        if (p.is_causal) visible = visible && key <= i + off;
        if (p.window > 0) visible = visible && key >= i + off + 1 - p.window;
        float s = 0.0f;
        const float* qr = sq + lr * d;
        const float* kr = sk + lane * kstride;
        for (int c = 0; c < d; ++c) s = fmaf(qr[c], kr[c], s);
        s *= p.scale;
        if (p.softcap != 0.0f) s = p.softcap * tanhf(s / p.softcap);
        const float x = visible ? s : NEG_INF;
        float mt = x;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
        const float m_new = fmaxf(m[r], mt);
        if (m_new == NEG_INF) continue;          // nothing visible yet (warp-uniform)
        const float alpha = expf(m[r] - m_new);  // exp(-inf) = 0 on the first visible tile
        const float pr = visible ? expf(x - m_new) : 0.0f;
        float ps = pr;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
        l[r] = l[r] * alpha + ps;
        m[r] = m_new;
#pragma unroll
        for (int u = 0; u < kChan; ++u) acc[r][u] *= alpha;
        for (int j = 0; j < nk; ++j) {
          const float pj = __shfl_sync(0xffffffffu, pr, j);
          const float* vr = sv + j * dv;
#pragma unroll
          for (int u = 0; u < kChan; ++u) {
            const int c = lane + 32 * u;
            if (c < dv) acc[r][u] = fmaf(pj, vr[c], acc[r][u]);
          }
        }
      }
    }

#pragma unroll
    for (int r = 0; r < kRowsPerWarp; ++r) {
      const int lr = warp * kRowsPerWarp + r;
      if (lr >= nrows) continue;
      const float inv = l[r] > 0.0f ? 1.0f / l[r] : 0.0f;
      float* orow = O + ((size_t)(item.q_start + row0 + lr) * p.H + hh) * dv;
#pragma unroll
      for (int u = 0; u < kChan; ++u) {
        const int c = lane + 32 * u;
        if (c < dv) orow[c] = acc[r][u] * inv;
      }
    }
  }
}

}  // namespace

cudaError_t launch_prefill_f32(const AttnParams& p, int num_sms, cudaStream_t s) {
  const size_t smem =
      sizeof(float) * (kF32TileTokens * p.d + kF32KeyTile * (p.d + 1) + kF32KeyTile * p.dv);
  cudaError_t e = cudaFuncSetAttribute(pva_prefill_f32_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(pva_prefill_f32_kernel, dim3(num_sms * 4), dim3(kWarps * 32), smem, s,
                          p);
}

}  // namespace pva
