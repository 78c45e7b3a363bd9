// bf16/f16 prefill on the 5th-generation tensor cores (tcgen05 + TMEM) with
// TMA-staged operands, for head sizes d = dv in {64, 128, 256}.
//
// The arithmetic is the page's (packed_varlen_attention.rs, stages 1-5:
// scale * q.k, optional softcap * tanh(score / softcap) before the mask, the
// tail-aligned causal frontier j <= i + L_kv - L_q, max-subtracted
// exponentials, zero rows when nothing is visible, weighted sum of V) but it
// streams over key tiles with a running maximum (online softmax), so no score
// matrix is ever stored.
//
// Work item = (sequence, query tile, kv head g).  The G = H/Hkv query heads
// that share kv head g are packed along the MMA's M dimension: a query tile
// holds m = floor(128 / G) tokens x G heads = up to 128 rows, so every K/V
// tile that is loaded serves all G heads (GQA reuse inside the CTA).
//
// Per CTA (persistent, one per SM, 192 threads):
//   warp 0      TMA producer: Q tile once per item, then K/V tiles into a
//               STAGES-deep ring (mbarrier full/empty pairs).
//   warp 1      MMA issuer (one thread) + TMEM owner: S = Q K^T into one of
//               two TMEM score buffers, O += P V into the TMEM accumulator.
//   warps 2..5  softmax / correction / epilogue: one thread per TMEM lane
//               (= MMA row).  Reads S with tcgen05.ld, applies scale,
//               softcap and masks, keeps the running max and sum, writes P
//               (16-bit) into shared memory in the 128-byte-swizzled layout
//               the MMA reads, rescales O in TMEM when the max grows by more
//               than 2^8 (lazily), and finally normalises O and stores the
//               rows that belong to the item.
//
// Key tiles beyond the causal frontier of an item's last row are never
// loaded; the diagonal tile and the ragged last tile are masked per element.
// Tiles that would run past the end of the packed buffers are shifted back
// so they end at the buffer's last row (columns/rows that belong to other
// positions are masked or discarded); tiles starting before row 0 are
// zero-filled by the TMA unit.  Nothing outside [0, cu[B]) rows is read.
#include "pva_device.cuh"
#include "pva_items.cuh"

namespace pva {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows > 2^8

template <int D>
struct TcCfg {
  static constexpr int BN = tc_block_n(D);
  static constexpr int STAGES = D == 64 ? 3 : 2;
  static constexpr int KCH = D / 64;              // 128-byte column chunks of a row
  static constexpr int Q_CHUNK = kTcRows * 128;   // bytes of one chunk of the Q tile
  static constexpr int Q_BYTES = KCH * Q_CHUNK;
  static constexpr int KV_CHUNK = BN * 128;       // bytes of one chunk of a K or V tile
  static constexpr int K_BYTES = KCH * KV_CHUNK;
  static constexpr int STAGE_BYTES = 2 * K_BYTES;  // K then V
  static constexpr int P_CHUNK = kTcRows * 128;   // 64 keys x 128 rows
  static constexpr int P_BYTES = (BN / 64) * P_CHUNK;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = Q_BYTES;
  static constexpr int OFF_P = OFF_KV + STAGES * STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BYTES;
  static constexpr int N_BARS = 16;
  static constexpr int SMEM = OFF_BAR + N_BARS * 8 + 1024;  // + alignment slack
  static constexpr int TMEM_COLS = 512;
  static constexpr int COL_S0 = 0, COL_S1 = BN, COL_O = 2 * BN;
  static_assert(2 * BN + D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct Bars {
  uint64_t q_full, q_empty, p_full, o_ready, o_free, drain;
  uint64_t s_full[2];
  uint64_t kv_full[4], kv_empty[4];
};

struct ItemGeom {
  PrefillItem it;
  int n_tiles;   // key tiles to visit (0: every row fully masked)
  int tile_q0;   // first packed token of the loaded Q tile (may be < q_start)
};

template <int D>
__device__ __forceinline__ ItemGeom item_geom(const AttnParams& p, const SchedHeader& h, int idx,
                                              int total_q) {
  ItemGeom g;
  g.it = decode_prefill_item(p, h, idx);
  const int hi = item_key_extent(g.it, h.tile_tokens, p.is_causal);
  g.n_tiles = (hi + TcCfg<D>::BN - 1) / TcCfg<D>::BN;
  const int want = g.it.q_start + g.it.t * h.tile_tokens;
  g.tile_q0 = min(want, total_q - h.tile_tokens);
  return g;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    pva_prefill_tc_kernel(AttnParams p, const __grid_constant__ CUtensorMap tmap_q,
                          const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v) {
  using C = TcCfg<D>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = smem + C::OFF_Q;
  uint8_t* sP = smem + C::OFF_P;
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = p.status;
  volatile int* abort = &s_abort;
  const int G = p.G;
  const int m_tok = kTcRows / G;  // tokens per query tile (one tile per item)
  const int total_q = p.cu_q[p.B];
  const int total_kv = p.cu_kv[p.B];

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->p_full, 128);
    mbar_init(&bars->o_ready, 1);
    mbar_init(&bars->o_free, 128);
    mbar_init(&bars->drain, 1);
    mbar_init(&bars->s_full[0], 1);
    mbar_init(&bars->s_full[1], 1);
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    fence_mbar_init();
  }
  // Rows of the Q tile beyond G*m are never written by the TMA unit; start
  // them (and everything else) from zeros so no stale bits reach the MMA.
  for (int i = threadIdx.x; i < C::Q_BYTES / 16; i += kThreads)
    reinterpret_cast<uint4*>(sQ)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) tmem_alloc<C::TMEM_COLS>(&s_tmem_base);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = s_tmem_base;
  wait_prior_grid();  // the scheduler's work lists are complete from here on
  allow_next_grid();
  const SchedHeader h = *reinterpret_cast<const SchedHeader*>(p.ws + kWsHeader);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&tmap_q);
      prefetch_tensor_map(&tmap_k);
      prefetch_tensor_map(&tmap_v);
      uint32_t q_cnt = 0, kv_cnt = 0;
      const uint32_t q_bytes = (uint32_t)C::KCH * (uint32_t)(G * m_tok) * 128u;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < h.n_items; idx += gridDim.x) {
        const ItemGeom ig = item_geom<D>(p, h, idx, total_q);
        if (ig.n_tiles == 0) continue;
        const int g = ig.it.unit;
        if (!(ok = mbar_wait(&bars->q_empty, (q_cnt & 1) ^ 1, abort, status))) break;
        mbar_arrive_expect_tx(&bars->q_full, q_bytes);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_load_3d(sQ + c * C::Q_CHUNK, &tmap_q, &bars->q_full, c * 64, g * G, ig.tile_q0);
        ++q_cnt;
        for (int j = 0; j < ig.n_tiles; ++j, ++kv_cnt) {
          const int st = kv_cnt % C::STAGES;
          const uint32_t use = kv_cnt / C::STAGES;
          if (!(ok = mbar_wait(&bars->kv_empty[st], (use & 1) ^ 1, abort, status))) break;
          uint8_t* sK = smem + C::OFF_KV + st * C::STAGE_BYTES;
          uint8_t* sV = sK + C::K_BYTES;
          const int k0 = min(ig.it.kv_start + j * BN, total_kv - BN);
          mbar_arrive_expect_tx(&bars->kv_full[st], (uint32_t)C::STAGE_BYTES);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c) {
            tma_load_3d(sK + c * C::KV_CHUNK, &tmap_k, &bars->kv_full[st], c * 64, g, k0);
            tma_load_3d(sV + c * C::KV_CHUNK, &tmap_v, &bars->kv_full[st], c * 64, g, k0);
          }
        }
      }
      // Drain: every copy this thread issued must land before the CTA exits.
      if (q_cnt) mbar_wait(&bars->q_full, (q_cnt - 1) & 1, abort, status);
      for (int s = 0; s < C::STAGES; ++s) {
        const uint32_t fills = kv_cnt > (uint32_t)s ? (kv_cnt - 1 - s) / C::STAGES + 1 : 0;
        if (fills) mbar_wait(&bars->kv_full[s], (fills - 1) & 1, abort, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16<T>(kTcRows, BN, false, false);
      constexpr uint32_t idesc_o = idesc_f16<T>(kTcRows, D, false, true);
      const uint32_t sQ_a = smem_u32(sQ), sP_a = smem_u32(sP);
      uint32_t q_cnt = 0, gt = 0, items = 0;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < h.n_items; idx += gridDim.x) {
        const ItemGeom ig = item_geom<D>(p, h, idx, total_q);
        const int n = ig.n_tiles;
        if (n == 0) continue;
        if (!(ok = mbar_wait(&bars->q_full, q_cnt & 1, abort, status))) break;
        tc_fence_after();
        for (int j = 0; ok && j <= n; ++j) {
          if (j < n) {
            const uint32_t T_ = gt + j;
            const int st = T_ % C::STAGES;
            if (!(ok = mbar_wait(&bars->kv_full[st], (T_ / C::STAGES) & 1, abort, status))) break;
            tc_fence_after();
            const uint32_t sK_a = smem_u32(smem + C::OFF_KV + st * C::STAGE_BYTES);
            const uint32_t d_s = tmem + ((T_ & 1) ? C::COL_S1 : C::COL_S0);
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint32_t koff = (kk & 3) * 32;
              const uint64_t a = sdesc_sw128(sQ_a + (kk >> 2) * C::Q_CHUNK + koff, 16, 1024);
              const uint64_t b = sdesc_sw128(sK_a + (kk >> 2) * C::KV_CHUNK + koff, 16, 1024);
              mma_ss(d_s, a, b, idesc_s, kk > 0 ? 1u : 0u);
            }
            mma_commit(&bars->s_full[T_ & 1]);
            if (j == n - 1) mma_commit(&bars->q_empty);
          }
          if (j > 0) {
            const uint32_t T_ = gt + j - 1;
            const int st = T_ % C::STAGES;
            if (j == 1 && !(ok = mbar_wait(&bars->o_free, (items & 1) ^ 1, abort, status))) break;
            if (!(ok = mbar_wait(&bars->p_full, T_ & 1, abort, status))) break;
            tc_fence_after();
            const uint32_t sV_a =
                smem_u32(smem + C::OFF_KV + st * C::STAGE_BYTES + C::K_BYTES);
#pragma unroll
            for (int kk = 0; kk < BN / 16; ++kk) {
              const uint64_t a =
                  sdesc_sw128(sP_a + (kk >> 2) * C::P_CHUNK + (kk & 3) * 32, 16, 1024);
              const uint64_t b = sdesc_sw128(sV_a + kk * 16 * 128, C::KV_CHUNK, 1024);
              mma_ss(tmem + C::COL_O, a, b, idesc_o, (j > 1 || kk > 0) ? 1u : 0u);
            }
            mma_commit(&bars->kv_empty[st]);
            mma_commit(&bars->o_ready);
          }
        }
        gt += n;
        ++q_cnt;
        ++items;
      }
      // Drain: all issued MMAs complete before TMEM is released.
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, abort, status);
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const float NEG_INF = __int_as_float(0xff800000);
    const bool capped = p.softcap != 0.0f;
    const float s_mul = capped ? p.scale / p.softcap : p.scale * kLog2e;
    const float cap_mul = p.softcap * kLog2e;
    uint32_t gt = 0, items = 0;
    bool ok = true;
    T* out = static_cast<T*>(p.out);

    for (int idx = blockIdx.x; ok && idx < h.n_items; idx += gridDim.x) {
      const ItemGeom ig = item_geom<D>(p, h, idx, total_q);
      const PrefillItem& it = ig.it;
      const int n = ig.n_tiles;
      const int tok = ig.tile_q0 + r / G;  // packed token of this row
      const int i = tok - it.q_start;       // its local query position
      const bool own = r < G * m_tok && i >= it.t * m_tok && i < min((it.t + 1) * m_tok, it.lq);
      const size_t orow = ((size_t)tok * p.H + (size_t)it.unit * G + (r % G)) * D;
      if (n == 0) {
        if (own) {
#pragma unroll
          for (int c = 0; c < D; c += 8)
            *reinterpret_cast<uint4*>(out + orow + c) = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      const int off = it.lkv - it.lq;
      const int row_hi = p.is_causal ? min(it.lkv, i + off + 1) : it.lkv;
      float m_used = NEG_INF, l = 0.0f;

      for (int j = 0; j < n; ++j) {
        const uint32_t T_ = gt + j;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[T_ & 1], (T_ >> 1) & 1, abort, status));
        if (!ok) break;
        tc_fence_after();
        float s[BN];
        {
          const uint32_t col = (T_ & 1) ? C::COL_S1 : C::COL_S0;
#pragma unroll
          for (int c = 0; c < BN; c += 32) {
            uint32_t v[32];
            tmem_ld32(t_lane + col + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) s[c + e] = __uint_as_float(v[e]);
          }
        }
        // visible columns [lo_c, hi_c) of this key tile
        const int k0 = min(it.kv_start + j * BN, total_kv - BN);
        const int base = k0 - it.kv_start;  // local key index of column 0
        const int lo_c = j * BN - base;
        const int hi_c = min((j + 1) * BN, row_hi) - base;
        float mt = NEG_INF;
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          float x = capped ? cap_mul * tanh_via_exp2(s[c] * s_mul) : s[c] * s_mul;
          x = (c >= lo_c && c < hi_c) ? x : NEG_INF;
          s[c] = x;
          mt = fmaxf(mt, x);
        }
        const float m_new = fmaxf(m_used, mt);
        float alpha = 1.0f;
        if (m_new > m_used + kRescaleThreshold) {
          alpha = ex2_approx(m_used - m_new);  // 0 when m_used is -inf
          m_used = m_new;
        }
        const float m_eff = m_used == NEG_INF ? 0.0f : m_used;
        float rs = 0.0f;
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          s[c] = ex2_approx(s[c] - m_eff);
          rs += s[c];
        }
        l = l * alpha + rs;

        if (j > 0) {
          // PV of the previous tile must be complete: it reads the P buffer
          // we are about to overwrite and accumulates into O.
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready, (T_ - 1) & 1, abort, status));
          if (!ok) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t v[32];
              tmem_ld32(t_lane + C::COL_O + c, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
              tmem_st32(t_lane + C::COL_O + c, v);
            }
            tmem_wait_st();
          }
        }
        // P (16-bit) -> shared memory, K-major, 128-byte swizzle: row r,
        // 16-byte chunk q of a 64-key half lands at chunk q ^ (r & 7).
#pragma unroll
        for (int c = 0; c < BN; c += 8) {
          uint4 w;
          w.x = pack2<T>(s[c + 0], s[c + 1]);
          w.y = pack2<T>(s[c + 2], s[c + 3]);
          w.z = pack2<T>(s[c + 4], s[c + 5]);
          w.w = pack2<T>(s[c + 6], s[c + 7]);
          const int half = c >> 6, q16 = (c & 63) >> 3;
          uint8_t* dst = sP + half * C::P_CHUNK + r * 128 + ((q16 ^ (r & 7)) << 4);
          *reinterpret_cast<uint4*>(dst) = w;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full);
      }
      if (!ok) break;

      // epilogue: O / l -> out (rows of this item only)
      const uint32_t T_last = gt + n - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready, T_last & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t v[32];
        tmem_ld32(t_lane + C::COL_O + c, v);
        tmem_wait_ld();
        if (own) {
#pragma unroll
          for (int e = 0; e < 32; e += 8) {
            uint4 w;
            w.x = pack2<T>(__uint_as_float(v[e + 0]) * inv, __uint_as_float(v[e + 1]) * inv);
            w.y = pack2<T>(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
            w.z = pack2<T>(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
            w.w = pack2<T>(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
            *reinterpret_cast<uint4*>(out + orow + c + e) = w;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free);
      gt += n;
      ++items;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<C::TMEM_COLS>(tmem);
}

template <typename T, int D>
cudaError_t launch_tc(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, int num_sms, cudaStream_t s) {
  constexpr int smem = TcCfg<D>::SMEM;
  auto kern = pva_prefill_tc_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, dim3(num_sms), dim3(kThreads), smem, s, p, tq, tk, tv);
}

}  // namespace

cudaError_t launch_prefill_tc(const AttnParams& p, int dtype, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv, int num_sms,
                              cudaStream_t s) {
  const bool bf = dtype == PVA_BF16;
  switch (p.d) {
    case 256:
      return bf ? launch_tc<__nv_bfloat16, 256>(p, tq, tk, tv, num_sms, s)
                : launch_tc<__half, 256>(p, tq, tk, tv, num_sms, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pva
