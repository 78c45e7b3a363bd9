// bf16/f16 prefill on tcgen05/TMEM for head sizes d = dv in {64, 128}: two
// 128-row query tiles per CTA share every K/V tile (paired tiles).
//
// Same arithmetic as pva_prefill_tc.cu (packed_varlen_attention.rs, stages
// 1-5, streamed as an online softmax).  The difference is the schedule: a
// work item covers 2m tokens (m = floor(128/G) tokens x G heads per tile), so
// each K/V tile is loaded once for 256 MMA rows, and the tensor core
// alternates between the two tiles: while softmax warpgroup 0 turns S0(j)
// into P0(j), the tensor core works on tile 1, and vice versa.
//
// Per CTA (persistent, one per SM, 320 threads):
//   warp 0      TMA producer: the item's two Q tiles, then K_j and V_j into a
//               ring of slots (K and V separately, so K_{j+1} can land while
//               V_j is still being read).
//   warp 1      MMA issuer + TMEM owner.  Order per key tile j:
//               PV0(j), S0(j+1), PV1(j), S1(j+1)  (S0(0), S1(0) up front).
//   warps 2..5  softmax / correction / epilogue for query tile 0
//   warps 6..9  the same for query tile 1
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+d), O1 after O0.
// P_t (16-bit, two per column) overwrites the first 64 columns of S_t once
// they have been read, and the P.V MMA takes its A operand from TMEM; the
// next S_t MMA is issued after that P.V MMA (tcgen05 MMAs of one thread run in
// issue order).  Shared memory (d = 128): Q0, Q1 32 KB each + 5 K/V slots of
// 32 KB.
#include "pva_device.cuh"
#include "pva_items.cuh"

namespace pva {
namespace {

constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxSlots = 12;

template <int D>
struct PairCfg {
  static constexpr int BN = 128;
  static constexpr int KCH = D / 64;
  static constexpr int Q_CHUNK = kTcRows * 128;       // 16 KB
  static constexpr int Q_TILE = KCH * Q_CHUNK;
  static constexpr int KV_CHUNK = BN * 128;           // 16 KB
  static constexpr int KV_TILE = KCH * KV_CHUNK;
  static constexpr int SLOTS = D == 128 ? 5 : 12;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = 2 * Q_TILE;
  static constexpr int OFF_BAR = OFF_RING + SLOTS * KV_TILE;
  static constexpr int SMEM = OFF_BAR + 512 + 1024;   // barriers + alignment slack
  static constexpr int TMEM_COLS = 512;
  static constexpr int COL_S = 0;        // + 128 * tile
  static constexpr int COL_O = 256;      // + D * tile
  static_assert(SLOTS <= kMaxSlots, "barrier array");
  static_assert(2 * BN + 2 * D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448 - 64, "shared memory budget");
};

struct PairBars {
  uint64_t q_full, q_empty, drain, pad;
  uint64_t s_full[2], p_full[2], o_ready[2], o_free[2];
  uint64_t ring_full[kMaxSlots], ring_empty[kMaxSlots];
};
static_assert(sizeof(PairBars) <= 512, "barrier block");

struct PairGeom {
  PrefillItem it;
  int n_tiles;  // key tiles (both query tiles visit the same ones)
  int q0;       // packed token of row-group 0 of query tile 0 (tile 1 = q0 + m)
};

__device__ __forceinline__ PairGeom pair_geom(const AttnParams& p, const SchedHeader& h, int idx,
                                              int total_q, int m) {
  PairGeom g;
  g.it = decode_prefill_item(p, h, idx);
  const int hi = item_key_extent(g.it, h.tile_tokens, p.is_causal);
  g.n_tiles = (hi + 127) / 128;
  const int want = g.it.q_start + g.it.t * h.tile_tokens;
  g.q0 = min(want, total_q - 2 * m);
  return g;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 1)
    pva_prefill_pair_kernel(AttnParams p, const __grid_constant__ CUtensorMap tmap_q,
                            const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v) {
  using C = PairCfg<D>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  PairBars* bars = reinterpret_cast<PairBars*>(smem + C::OFF_BAR);
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = p.status;
  volatile int* abort = &s_abort;
  const int G = p.G;
  const int m_tok = kTcRows / G;  // tokens per query tile (the item covers 2 m)
  const int total_q = p.cu_q[p.B];
  const int total_kv = p.cu_kv[p.B];

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->drain, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_ready[t], 1);
      mbar_init(&bars->o_free[t], 128);
    }
    for (int s = 0; s < C::SLOTS; ++s) {
      mbar_init(&bars->ring_full[s], 1);
      mbar_init(&bars->ring_empty[s], 1);
    }
    fence_mbar_init();
  }
  // Rows of the Q tiles beyond G*m are never written by the TMA unit; start
  // them from zeros so no stale bits reach the MMA.
  for (int i = threadIdx.x; i < 2 * C::Q_TILE / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + C::OFF_Q)[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  if (warp == 1) tmem_alloc<C::TMEM_COLS>(&s_tmem_base);
  if (warp == 0 && lane == 0) {
    prefetch_tensor_map(&tmap_q);
    prefetch_tensor_map(&tmap_k);
    prefetch_tensor_map(&tmap_v);
  }
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
      uint32_t items = 0, loads = 0;
      const uint32_t q_bytes = 2u * C::KCH * (uint32_t)(G * m_tok) * 128u;
      bool ok = true;
      for (int idx = blockIdx.x; ok && idx < h.n_items; idx += gridDim.x) {
        const PairGeom pg = pair_geom(p, h, idx, total_q, m_tok);
        if (pg.n_tiles == 0) continue;
        const int g = pg.it.unit;
        if (!(ok = mbar_wait(&bars->q_empty, (items & 1) ^ 1, abort, status))) break;
        mbar_arrive_expect_tx(&bars->q_full, q_bytes);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_load_3d(smem + C::OFF_Q + t * C::Q_TILE + c * C::Q_CHUNK, &tmap_q, &bars->q_full,
                        c * 64, g * G, pg.q0 + t * m_tok);
        ++items;
        for (int j = 0; ok && j < pg.n_tiles; ++j) {
          const int k0 = min(pg.it.kv_start + j * BN, total_kv - BN);
#pragma unroll
          for (int kv = 0; kv < 2; ++kv, ++loads) {
            const int sl = loads % C::SLOTS;
            if (!(ok = mbar_wait(&bars->ring_empty[sl], ((loads / C::SLOTS) & 1) ^ 1, abort,
                                 status)))
              break;
            uint8_t* dst = smem + C::OFF_RING + sl * C::KV_TILE;
            mbar_arrive_expect_tx(&bars->ring_full[sl], (uint32_t)C::KV_TILE);
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_3d(dst + c * C::KV_CHUNK, kv ? &tmap_v : &tmap_k, &bars->ring_full[sl],
                          c * 64, g, k0);
          }
        }
      }
      // Drain: every copy this thread issued must land before the CTA exits.
      if (items) mbar_wait(&bars->q_full, (items - 1) & 1, abort, status);
      for (int s = 0; s < C::SLOTS; ++s) {
        const uint32_t fills = loads > (uint32_t)s ? (loads - 1 - s) / C::SLOTS + 1 : 0;
        if (fills) mbar_wait(&bars->ring_full[s], (fills - 1) & 1, abort, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16<T>(kTcRows, BN, false, false);
      constexpr uint32_t idesc_o = idesc_f16<T>(kTcRows, D, false, true);
      const uint32_t sQ = smem_u32(smem + C::OFF_Q);
      const uint32_t sRing = smem_u32(smem + C::OFF_RING);
      uint32_t items = 0, loads = 0, tiles = 0;  // tiles: key tiles done (per query tile)
      bool ok = true;
      auto issue_s = [&](int t, uint32_t kslot) {
        const uint32_t q_a = sQ + t * C::Q_TILE;
        const uint32_t k_a = sRing + kslot * C::KV_TILE;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          mma_ss(tmem + C::COL_S + t * 128,
                 sdesc_sw128(q_a + (kk >> 2) * C::Q_CHUNK + off, 16, 1024),
                 sdesc_sw128(k_a + (kk >> 2) * C::KV_CHUNK + off, 16, 1024), idesc_s,
                 kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[t]);
      };
      auto issue_pv = [&](int t, uint32_t vslot, bool first) {
        const uint32_t v_a = sRing + vslot * C::KV_TILE;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma_ts(tmem + C::COL_O + t * D, tmem + C::COL_S + t * 128 + kk * 8,
                 sdesc_sw128(v_a + kk * 16 * 128, C::KV_CHUNK, 1024), idesc_o,
                 (!first || kk > 0) ? 1u : 0u);
        mma_commit(&bars->o_ready[t]);
      };
      auto wait_slot = [&](uint32_t L) -> bool {
        const bool r = mbar_wait(&bars->ring_full[L % C::SLOTS], (L / C::SLOTS) & 1, abort, status);
        tc_fence_after();
        return r;
      };
      for (int idx = blockIdx.x; ok && idx < h.n_items; idx += gridDim.x) {
        const PairGeom pg = pair_geom(p, h, idx, total_q, m_tok);
        const int n = pg.n_tiles;
        if (n == 0) continue;
        if (!(ok = mbar_wait(&bars->q_full, items & 1, abort, status))) break;
        tc_fence_after();
        // key tile j lives in load slots (loads + 2j) (K) and (loads + 2j + 1) (V)
        if (!(ok = wait_slot(loads))) break;
        issue_s(0, loads % C::SLOTS);
        issue_s(1, loads % C::SLOTS);
        mma_commit(&bars->ring_empty[loads % C::SLOTS]);
        if (n == 1) mma_commit(&bars->q_empty);
        for (int j = 0; ok && j < n; ++j) {
          const uint32_t Lk = loads + 2 * j, Lv = Lk + 1, Lk1 = Lk + 2;
          const uint32_t T_ = tiles + j;
          // PV0(j)
          if (j == 0 && !(ok = mbar_wait(&bars->o_free[0], (items & 1) ^ 1, abort, status))) break;
          if (!(ok = mbar_wait(&bars->p_full[0], T_ & 1, abort, status))) break;
          if (!(ok = wait_slot(Lv))) break;
          issue_pv(0, Lv % C::SLOTS, j == 0);
          // S0(j+1)
          if (j + 1 < n) {
            if (!(ok = wait_slot(Lk1))) break;
            issue_s(0, Lk1 % C::SLOTS);
          }
          // PV1(j)
          if (j == 0 && !(ok = mbar_wait(&bars->o_free[1], (items & 1) ^ 1, abort, status))) break;
          if (!(ok = mbar_wait(&bars->p_full[1], T_ & 1, abort, status))) break;
          tc_fence_after();
          issue_pv(1, Lv % C::SLOTS, j == 0);
          mma_commit(&bars->ring_empty[Lv % C::SLOTS]);
          // S1(j+1)
          if (j + 1 < n) {
            issue_s(1, Lk1 % C::SLOTS);
            mma_commit(&bars->ring_empty[Lk1 % C::SLOTS]);
            if (j + 2 == n) mma_commit(&bars->q_empty);
          }
        }
        loads += 2 * n;
        tiles += n;
        ++items;
      }
      // Drain: all issued MMAs complete before TMEM is released.
      mma_commit(&bars->drain);
      mbar_wait(&bars->drain, 0, abort, status);
    }
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int tq = warp >= 6 ? 1 : 0;  // query tile of this warpgroup
    const int quarter = warp & 3;      // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t col_s = C::COL_S + tq * 128, col_o = C::COL_O + tq * D;
    const float NEG_INF = __int_as_float(0xff800000);
    const bool capped = p.softcap != 0.0f;
    const float s_mul = capped ? p.scale / p.softcap : p.scale * kLog2e;
    const float cap_mul = p.softcap * kLog2e;
    const bool up = p.scale > 0.0f;  // direction of the (monotone) score transform
    uint32_t tiles = 0;
    bool ok = true;
    T* out = static_cast<T*>(p.out);

    for (int idx = blockIdx.x; ok && idx < h.n_items; idx += gridDim.x) {
      const PairGeom pg = pair_geom(p, h, idx, total_q, m_tok);
      const PrefillItem& it = pg.it;
      const int n = pg.n_tiles;
      const int tok = pg.q0 + tq * m_tok + r / G;
      const int i = tok - it.q_start;
      const int first = it.t * h.tile_tokens;
      const bool own = r < G * m_tok && i >= first && i < min(first + h.tile_tokens, it.lq);
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
        const uint32_t T_ = tiles + j;
        ok = __all_sync(0xffffffffu, mbar_wait(&bars->s_full[tq], T_ & 1, abort, status));
        if (!ok) break;
        tc_fence_after();
        const int k0 = min(it.kv_start + j * BN, total_kv - BN);
        const int base = k0 - it.kv_start;  // local key index of column 0
        const int lo_c = j * BN - base;     // visible columns [lo_c, hi_c)
        const int hi_c = min((j + 1) * BN, row_hi) - base;
        const bool full_tile = __all_sync(0xffffffffu, lo_c <= 0 && hi_c >= BN);
        // Pass 1: extreme raw score over the visible columns.  The score
        // transform (scale, then optional softcap) is monotone -- increasing
        // for scale > 0, decreasing for scale < 0 -- so the row max of the
        // transformed scores is the transform of this extreme.
        float ext = up ? NEG_INF : -NEG_INF;
#pragma unroll
        for (int c = 0; c < BN; c += 64) {
          uint32_t va[32], vb[32];
          tmem_ld32(t_lane + col_s + c, va);
          tmem_ld32(t_lane + col_s + c + 32, vb);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            float x = __uint_as_float(e < 32 ? va[e] : vb[e - 32]);
            if (!full_tile && (c + e < lo_c || c + e >= hi_c)) x = up ? NEG_INF : -NEG_INF;
            ext = up ? fmaxf(ext, x) : fminf(ext, x);
          }
        }
        const float mt = (ext == NEG_INF || ext == -NEG_INF)
                             ? NEG_INF
                             : (capped ? cap_mul * tanh_via_exp2(ext * s_mul) : ext * s_mul);
        const float m_new = fmaxf(m_used, mt);
        float alpha = 1.0f;
        if (m_new > m_used + kRescaleThreshold) {
          alpha = ex2_approx(m_used - m_new);  // 0 when m_used is -inf
          m_used = m_new;
        }
        const float m_eff = m_used == NEG_INF ? 0.0f : m_used;
        if (j > 0) {
          // PV of the previous tile must be complete before O is rescaled.
          ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready[tq], (T_ - 1) & 1, abort, status));
          if (!ok) break;
          tc_fence_after();
          if (__any_sync(0xffffffffu, alpha != 1.0f)) {
#pragma unroll 1
            for (int c = 0; c < D; c += 32) {
              uint32_t v[32];
              tmem_ld32(t_lane + col_o + c, v);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
              tmem_st32(t_lane + col_o + c, v);
            }
          }
        }
        // Pass 2: p = 2^(x - m), row sum, P (16-bit pairs) into TMEM over the
        // S columns already read: columns [c, c+32) of S become P columns
        // [c/2, c/2 + 16).
        float rs = 0.0f;
#pragma unroll
        for (int c = 0; c < BN; c += 64) {
          uint32_t va[32], vb[32];
          tmem_ld32(t_lane + col_s + c, va);
          tmem_ld32(t_lane + col_s + c + 32, vb);
          tmem_wait_ld();
          uint32_t pw[32];
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            float pr[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int cc = e + u;
              const float sraw = __uint_as_float(cc < 32 ? va[cc] : vb[cc - 32]);
              float x = capped ? cap_mul * tanh_via_exp2(sraw * s_mul) - m_eff
                               : fmaf(sraw, s_mul, -m_eff);
              if (!full_tile && (c + cc < lo_c || c + cc >= hi_c)) x = NEG_INF;
              pr[u] = ex2_approx(x);
              rs += pr[u];
            }
            pw[e >> 1] = pack2<T>(pr[0], pr[1]);
          }
          uint32_t lo16[16], hi16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            lo16[e] = pw[e];
            hi16[e] = pw[16 + e];
          }
          tmem_st16(t_lane + col_s + (c >> 1), lo16);
          tmem_st16(t_lane + col_s + (c >> 1) + 16, hi16);
        }
        tmem_wait_st();
        l = l * alpha + rs;
        tc_fence_before();
        mbar_arrive(&bars->p_full[tq]);
      }
      if (!ok) break;

      // epilogue: O / l -> out (rows of this item only)
      const uint32_t T_last = tiles + n - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(&bars->o_ready[tq], T_last & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        uint32_t v[32];
        tmem_ld32(t_lane + col_o + c, v);
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
      mbar_arrive(&bars->o_free[tq]);
      tiles += n;
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<C::TMEM_COLS>(tmem);
}

template <typename T, int D>
cudaError_t launch_pair(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, int num_sms, cudaStream_t s) {
  constexpr int smem = PairCfg<D>::SMEM;
  auto kern = pva_prefill_pair_kernel<T, D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, dim3(num_sms), dim3(kThreads), smem, s, p, tq, tk, tv);
}

}  // namespace

cudaError_t launch_prefill_pair(const AttnParams& p, int dtype, const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv, int num_sms,
                                cudaStream_t s) {
  const bool bf = dtype == PVA_BF16;
  switch (p.d) {
    case 64:
      return bf ? launch_pair<__nv_bfloat16, 64>(p, tq, tk, tv, num_sms, s)
                : launch_pair<__half, 64>(p, tq, tk, tv, num_sms, s);
    case 128:
      return bf ? launch_pair<__nv_bfloat16, 128>(p, tq, tk, tv, num_sms, s)
                : launch_pair<__half, 128>(p, tq, tk, tv, num_sms, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pva
