// bf16/f16 prefill on the 5th-generation tensor cores (tcgen05 + TMEM) with
// TMA-staged operands, one 128-row query tile per CTA, for the head sizes the
// paired kernel does not take: (d, dv) = (256, 256), (192, 192), (192, 128)
// (q.k wider than v, as in multi-head latent attention) and (96, 96).  A head
// size that is not a multiple of 64 is loaded in 64-column boxes whose tail
// lies outside the tensor and reads the TMA zero fill; the MMAs never touch it.
//
// The arithmetic is the page's (packed_varlen_attention.rs, stages 1-5:
// scale * q.k, optional softcap * tanh(score / softcap) before the mask, the
// tail-aligned causal frontier j <= i + L_kv - L_q, max-subtracted
// exponentials, zero rows when nothing is visible, weighted sum of V) but it
// streams over key tiles of 64 keys with a running maximum (online softmax),
// so no score matrix is ever stored.
//
// Work item = (sequence, query tile of m = floor(128/G) tokens x G heads, kv
// head g): every K/V tile loaded serves all G query heads sharing it.
//
// Per CTA (persistent, one per SM, 192 threads):
//   warp 0      TMA producer: draws work items from a device-wide counter,
//               publishes each decoded item through a shared-memory ring, and
//               loads the Q tile, then K_j and V_j, into one ring of 7 to 14
//               slots (the Q tile takes 2 or 3 slots).
//   warp 1      MMA issuer + TMEM owner.  S = Q K^T takes Q from TMEM and K
//               from shared memory, so each S MMA reads only its 64 K rows
//               from shared memory.  S is double-buffered in TMEM (S(j) in
//               buffer j & 1), so S(j+1) runs while tile j is being
//               exponentiated; P(j) (16-bit pairs) overwrites S(j)'s buffer and
//               feeds O += P V with A taken from TMEM; S(j+2) reuses the buffer
//               after that MMA (tcgen05 MMAs of one thread run in issue order).
//   warps 2..5  softmax / correction / epilogue, one thread per TMEM lane;
//               they also move each Q tile from its ring slots into TMEM,
//               the next item's before the current item's epilogue.
// TMEM: S buffers [0,64) and [64,128), O [128,128+dv), Q [128+dv,
// 128+dv+d/2) (512 columns at d = dv = 256).
//
// Softcap: tanh(t) of the scaled score t = s * scale / softcap comes from its
// Maclaurin series t - t^3/3 + 2t^5/15 (error < 3.3e-6 for |t| <= 1/4, i.e.
// below 2.4e-4 in the base-2 exponent at softcap 50) with the softcap folded
// into the coefficients, on the FMA pipe, whenever every score of the warp's
// tile has |t| <= 1/4; otherwise from the identity
// tanh(t) = 1 - 2 / (exp(2t) + 1).
//
// Softmax per tile in two passes: the row extreme of the raw scores (the
// score transform is monotone), then the exponentials against the running
// maximum, which is raised (and O rescaled) only when it grows by more than
// 2^8.
#include "pva_device.cuh"
#include "pva_items.cuh"

namespace pva {
namespace {

constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O when the max grows > 2^8
constexpr int kItemSlots = 4;
constexpr int kSoftmaxWarps = 4;
constexpr float kPolyLimit = 0.25f;         // |t| range of the tanh series

template <int DQK, int DV>
struct TcCfg {
  static_assert(DQK % 32 == 0 && DV % 32 == 0 && DQK <= 256 && DV <= 256, "head sizes");
  static constexpr int BN = 64;
  static constexpr int KCH = (DQK + 63) / 64;     // 128-byte column chunks of a q/k row
  static constexpr int VCH = (DV + 63) / 64;      // the same for a v row
  static constexpr int Q_CHUNK = kTcRows * 128;   // bytes of one chunk of the Q tile
  static constexpr int KV_CHUNK = BN * 128;       // bytes of one chunk of a K or V tile
  static constexpr int K_BYTES = KCH * KV_CHUNK;
  static constexpr int V_BYTES = VCH * KV_CHUNK;
  static constexpr int KV_TILE = K_BYTES > V_BYTES ? K_BYTES : V_BYTES;  // one ring slot
  // The Q tile passes through the K/V ring on its way to TMEM: Q_PER_SLOT of
  // its 64-column chunks per slot, Q_SLOTS slots per tile.
  static constexpr int Q_PER_SLOT = KV_TILE / Q_CHUNK;
  static_assert(Q_PER_SLOT >= 1, "a Q chunk fits a ring slot");
  static constexpr int Q_SLOTS = (KCH + Q_PER_SLOT - 1) / Q_PER_SLOT;
  // As many ring slots as shared memory holds (at most 16): 7 at d = dv =
  // 256, 9 at d = 192, 14 at d = 96.  The loads in flight per SM are bounded
  // by the ring: a deeper ring starts each load earlier before its tile is
  // needed, which is what hides the L2 / DRAM latency.
  // Output staging for the epilogue's tensor stores: 4 KB per softmax warp
  // (its 32 rows x 64 columns), at dv <= 192 only (d = dv = 256 keeps the
  // ring slot: its items are long and its epilogue rare).
  static constexpr int STAGE_BYTES = DV <= 192 ? 4 * 4096 : 0;
  static constexpr int SLOTS_FIT = (232448 - 64 - 2048 - STAGE_BYTES) / KV_TILE;
  static constexpr int SLOTS = SLOTS_FIT < 16 ? SLOTS_FIT : 16;
  static_assert(SLOTS >= Q_SLOTS + 2, "K/V ring depth");
  static constexpr int OFF_RING = 0;
  static constexpr int OFF_STAGE = OFF_RING + SLOTS * KV_TILE;
  static constexpr int OFF_BAR = OFF_STAGE + STAGE_BYTES;
  static constexpr int SMEM = OFF_BAR + 1024 + 1024;  // barriers/items + alignment slack
  static constexpr int TMEM_COLS = 512;
  static constexpr int COL_S = 0;                 // + BN * buffer
  static constexpr int COL_O = 2 * BN;
  // Q as the A operand of S = Q K^T: row r in lane r, dims (2c, 2c+1) as a
  // 16-bit pair in column COL_Q + c
  static constexpr int COL_Q = COL_O + DV;
  static_assert(COL_Q + DQK / 2 <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448 - 64, "shared memory budget");
};

struct ItemSlot {
  int q_start, kv_start, lq, lkv;
  int t, unit, n_tiles, q0;
  int last;
  int jb;  // first key tile (a local window skips the ones before)
  int pad[2];
};

struct Bars {
  uint64_t q_tmem, o_ready, o_done, o_free, drain;
  uint64_t s_full[2], p_full[2];
  uint64_t ring_full[16], ring_empty[16];
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  ItemSlot items[kItemSlots];
};
static_assert(sizeof(Bars) <= 1024, "barrier block");

__device__ __forceinline__ float col32(const uint32_t (&va)[32], const uint32_t (&vb)[32], int e) {
  return __uint_as_float(e < 32 ? va[e] : vb[e - 32]);
}

// Extreme raw scores (max, and min for the softcap range test) of a 64-column
// tile; MASKED skips the columns outside [lo_c, hi_c).
template <bool MASKED>
__device__ __forceinline__ void extremes64(const uint32_t (&va)[32], const uint32_t (&vb)[32],
                                           int lo_c, int hi_c, float& mx, float& mn) {
  const float ninf = __int_as_float(0xff800000), pinf = __int_as_float(0x7f800000);
  float a[2] = {ninf, ninf}, b[2] = {pinf, pinf};
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    const float x0 = col32(va, vb, e), x1 = col32(va, vb, e + 1);
    const bool v0 = !MASKED || (e >= lo_c && e < hi_c);
    const bool v1 = !MASKED || (e + 1 >= lo_c && e + 1 < hi_c);
    a[(e >> 1) & 1] = fmax3f(a[(e >> 1) & 1], v0 ? x0 : ninf, v1 ? x1 : ninf);
    b[(e >> 1) & 1] = fmin3f(b[(e >> 1) & 1], v0 ? x0 : pinf, v1 ? x1 : pinf);
  }
  mx = fmaxf(a[0], a[1]);
  mn = fminf(b[0], b[1]);
}

// 2^(x - m) over the 64 columns, row sum, P packed as 16-bit pairs, where x
// is the scaled (MODE 0) or softcapped score in base-2 units.  MODE 1: A *
// tanh(u) for |u| <= 1/4 from the first three terms of the tanh series,
// u - u^3/3 + 2u^5/15, with A folded into the coefficients (u * (A + w *
// (-A/3 + w * 2A/15)), w = u^2); the series alternates with falling terms,
// so the error is below the next one, 17/315 |u|^7 < 3.3e-6.  MODE 2: tanh
// from exp/rcp.
template <typename T, int MODE, bool MASKED>
__device__ __forceinline__ float exp64(const uint32_t (&va)[32], const uint32_t (&vb)[32],
                                       int lo_c, int hi_c, float s_mul, float cap_mul,
                                       float m_eff, uint32_t (&pw)[32]) {
  const float2 z = make_float2(0.0f, 0.0f);
  const float2 mul2 = make_float2(s_mul, s_mul), neg_m = make_float2(-m_eff, -m_eff);
  const float2 a2 = make_float2(cap_mul, cap_mul);
  const float2 c1 = make_float2(cap_mul * (-1.0f / 3.0f), cap_mul * (-1.0f / 3.0f));
  const float2 c2 = make_float2(cap_mul * (2.0f / 15.0f), cap_mul * (2.0f / 15.0f));
  float2 acc[2] = {z, z};
#pragma unroll
  for (int e = 0; e < 64; e += 2) {
    const float2 s = make_float2(col32(va, vb, e), col32(va, vb, e + 1));
    float2 x;
    if (MODE == 0) {
      x = ffma2(s, mul2, neg_m);
    } else if (MODE == 1) {
      const float2 u = ffma2(s, mul2, z);
      const float2 w = ffma2(u, u, z);
      x = ffma2(u, ffma2(w, ffma2(w, c2, c1), a2), neg_m);
    } else {
      x.x = fmaf(cap_mul, tanh_via_exp2(s.x * s_mul), -m_eff);
      x.y = fmaf(cap_mul, tanh_via_exp2(s.y * s_mul), -m_eff);
    }
    if (MASKED) {
      const float ninf = __int_as_float(0xff800000);
      x.x = (e >= lo_c && e < hi_c) ? x.x : ninf;
      x.y = (e + 1 >= lo_c && e + 1 < hi_c) ? x.y : ninf;
    }
    const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    acc[(e >> 1) & 1] = fadd2(acc[(e >> 1) & 1], p);
    pw[e >> 1] = pack2<T>(p.x, p.y);
  }
  const float2 r = fadd2(acc[0], acc[1]);
  return r.x + r.y;
}

template <typename T, int DQK, int DV, bool CAP>
__global__ void __launch_bounds__(kThreads, 1)
    pva_prefill_tc_kernel(AttnParams p, const __grid_constant__ CUtensorMap tmap_q,
                          const __grid_constant__ CUtensorMap tmap_k,
                          const __grid_constant__ CUtensorMap tmap_v,
                          const __grid_constant__ CUtensorMap tmap_o) {
  using C = TcCfg<DQK, DV>;
  constexpr int BN = C::BN;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
  __shared__ uint32_t s_tmem_base;
  __shared__ int s_abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = p.status;
  volatile int* abort = &s_abort;
  const int G = p.G;
  const int m_tok = kTcRows / G;  // tokens per query tile (one tile per item)
  const int total_q = p.cu_q[p.B];
  const int total_kv = kv_tile_end(p);

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bars->q_tmem, 32 * kSoftmaxWarps);
    mbar_init(&bars->o_ready, 1);
    mbar_init(&bars->o_done, 1);
    mbar_init(&bars->o_free, 32 * kSoftmaxWarps);
    mbar_init(&bars->drain, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->s_full[b], 1);
      mbar_init(&bars->p_full[b], 32 * kSoftmaxWarps);
    }
    for (int s = 0; s < C::SLOTS; ++s) {
      mbar_init(&bars->ring_full[s], 1);
      mbar_init(&bars->ring_empty[s], 1);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 1 + kSoftmaxWarps);
    }
    fence_mbar_init();
  }
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const SchedHeader h = *reinterpret_cast<const SchedHeader*>(p.ws + kWsHeader);
      uint32_t loads = 0, published = 0;
      const uint32_t q_chunk_bytes = (uint32_t)(G * m_tok) * 128u;
      bool ok = true;
      auto publish = [&](const ItemSlot& v) -> bool {
        const int sl = published % kItemSlots;
        if (!mbar_wait<false>(&bars->item_empty[sl], ((published / kItemSlots) & 1) ^ 1, abort, status))
          return false;
        bars->items[sl] = v;
        mbar_arrive(&bars->item_full[sl]);
        ++published;
        return true;
      };
      // Items are drawn from a device-wide counter (zeroed by the scheduler):
      // a CTA takes the next item of the longest-first list when it is ready
      // for one, which balances uneven item costs across the persistent grid.
      // The next index is taken as soon as the current item starts, and the
      // next item is decoded once the current item's first loads are out, so
      // both latencies overlap the current item instead of delaying the next
      // publish.
      int* next_item = p.ws + WsLayout{p.B, p.Hkv}.counters();
      int idx = atomicAdd(next_item, 1);
      PrefillItem it{};
      if (idx < h.n_items) it = decode_prefill_item(p, h, idx, true);
      while (ok && idx < h.n_items) {
        const int idx_next = idx + 1 < h.n_items ? atomicAdd(next_item, 1) : h.n_items;
        PrefillItem it_next = it;
        bool decoded = idx_next >= h.n_items;
        const int hi = item_key_extent(it, h.tile_tokens, p.is_causal);
        ItemSlot v;
        v.q_start = it.q_start;
        v.kv_start = it.kv_start;
        v.lq = it.lq;
        v.lkv = it.lkv;
        v.t = it.t;
        v.unit = it.unit;
        v.jb = item_key_begin(it, h.tile_tokens, p.window) / BN;
        v.n_tiles = max(0, (hi + BN - 1) / BN - v.jb);
        v.q0 = min(it.q_start + it.t * h.tile_tokens, total_q - m_tok);
        v.last = 0;
        if (!(ok = publish(v))) break;
        if (v.n_tiles > 0) {
          const int g = v.unit;
          // the Q tile: Q_PER_SLOT chunks in each of the next Q_SLOTS slots
          for (int qs = 0; ok && qs < C::Q_SLOTS; ++qs, ++loads) {
            const int sl = loads % C::SLOTS;
            if (!(ok = mbar_wait<false>(&bars->ring_empty[sl], ((loads / C::SLOTS) & 1) ^ 1, abort,
                                        status)))
              break;
            const int c_lo = qs * C::Q_PER_SLOT, c_hi = min(C::KCH, c_lo + C::Q_PER_SLOT);
            mbar_arrive_expect_tx(&bars->ring_full[sl], (uint32_t)(c_hi - c_lo) * q_chunk_bytes);
            for (int c = c_lo; c < c_hi; ++c)
              tma_load_3d(smem + C::OFF_RING + sl * C::KV_TILE + (c - c_lo) * C::Q_CHUNK, &tmap_q,
                          &bars->ring_full[sl], c * 64, g * G, v.q0);
          }
          for (int j = 0; ok && j < v.n_tiles; ++j) {
            const int k0 = min(v.kv_start + (v.jb + j) * BN,
                               key_tile_limit(p, v.kv_start, v.lkv, total_kv) - BN);
#pragma unroll
            for (int kv = 0; kv < 2; ++kv, ++loads) {
              const int sl = loads % C::SLOTS;
              if (!(ok = mbar_wait<false>(&bars->ring_empty[sl], ((loads / C::SLOTS) & 1) ^ 1, abort,
                                   status)))
                break;
              uint8_t* dst = smem + C::OFF_RING + sl * C::KV_TILE;
              mbar_arrive_expect_tx(&bars->ring_full[sl],
                                    (uint32_t)(kv ? C::V_BYTES : C::K_BYTES));
              const int nch = kv ? C::VCH : C::KCH;
              for (int c = 0; c < nch; ++c)
                load_kv_box(dst + c * C::KV_CHUNK, kv ? &tmap_v : &tmap_k, &bars->ring_full[sl], p,
                            c * 64, it.b, g, v.kv_start, k0);
            }
            if (!decoded) {
              it_next = decode_prefill_item(p, h, idx_next, true);
              decoded = true;
            }
          }
        }
        if (!ok) break;
        if (!decoded) it_next = decode_prefill_item(p, h, idx_next, true);
        idx = idx_next;
        it = it_next;
      }
      if (ok) {
        ItemSlot v{};
        v.last = 1;
        publish(v);
      }
      // Drain: every copy this thread issued must land before the CTA exits.
      for (int s = 0; s < C::SLOTS; ++s) {
        const uint32_t fills = loads > (uint32_t)s ? (loads - 1 - s) / C::SLOTS + 1 : 0;
        if (fills) mbar_wait<false>(&bars->ring_full[s], (fills - 1) & 1, abort, status);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the loop and waits; one elected lane issues.
    const bool leader = elect_sync();
    constexpr uint32_t idesc_s = idesc_f16<T>(kTcRows, BN, false, false);
    constexpr uint32_t idesc_o = idesc_f16<T>(kTcRows, DV, false, true);
    // Base descriptors, built once: the issue loops only add constants.
    const uint64_t kdesc = sdesc_sw128(smem_u32(smem + C::OFF_RING), 16, 1024);
    const uint64_t vdesc = sdesc_sw128(smem_u32(smem + C::OFF_RING), C::KV_CHUNK, 1024);
    uint32_t q_cnt = 0, loads = 0, gt = 0, items = 0, taken = 0;  // q_cnt: Q tiles in TMEM
    bool ok = true;
    auto commit = [&](uint64_t* bar) {
      if (leader) mma_commit(bar);
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(bar, parity, abort, status));
    };
    auto wait_slot = [&](uint32_t L) -> bool {
      const bool r = wait(&bars->ring_full[L % C::SLOTS], (L / C::SLOTS) & 1);
      tc_fence_after();
      return r;
    };
    // S for global key tile T_ into buffer T_ & 1 from the K in load slot L
    auto issue_s = [&](uint32_t T_, uint32_t L) {
      const uint64_t ka = sdesc_advance(kdesc, (L % C::SLOTS) * C::KV_TILE);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < DQK / 16; ++kk) {
          const uint32_t off = (kk & 3) * 32;
          mma_ts(tmem + C::COL_S + (T_ & 1) * BN, tmem + C::COL_Q + kk * 8,
                 sdesc_advance(ka, (kk >> 2) * C::KV_CHUNK + off), idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[T_ & 1]);
        mma_commit(&bars->ring_empty[L % C::SLOTS]);  // K no longer needed once done
      }
    };
    while (ok) {
      const int isl = taken % kItemSlots;
      if (!(ok = wait(&bars->item_full[isl], (taken / kItemSlots) & 1))) break;
      const int n = bars->items[isl].n_tiles, last = bars->items[isl].last;
      __syncwarp();
      if (leader) mbar_arrive(&bars->item_empty[isl]);
      ++taken;
      if (last) break;
      if (n == 0) continue;
      // Q is in TMEM once every softmax thread has copied its share; its
      // ring slots are free from then on.
      if (!(ok = wait(&bars->q_tmem, q_cnt & 1))) break;
      tc_fence_after();
      if (leader) {
        for (int qs = 0; qs < C::Q_SLOTS; ++qs) mbar_arrive(&bars->ring_empty[(loads + qs) % C::SLOTS]);
      }
      loads += C::Q_SLOTS;
      // key tile j: K in load slot loads + 2j, V in loads + 2j + 1
      for (int j = 0; ok && j < 2 && j < n; ++j) {
        if (!(ok = wait_slot(loads + 2 * j))) break;
        issue_s(gt + j, loads + 2 * j);
      }
      if (!ok) break;
      for (int j = 0; ok && j < n; ++j) {
        const uint32_t T_ = gt + j, Lv = loads + 2 * j + 1;
        // P.V(j) needs V_j and P(j) only.  K_{j+2} is waited for only after
        // P.V(j) is issued: its ring slot is the one used SLOTS loads before,
        // so its load starts late, and waiting for it first would hold P.V(j)
        // -- and with it the slot of the load after -- behind a load latency.
        if (!(ok = wait_slot(Lv))) break;
        if (j == 0 && !(ok = wait(&bars->o_free, (items & 1) ^ 1))) break;
        if (!(ok = wait(&bars->p_full[T_ & 1], (T_ >> 1) & 1))) break;
        tc_fence_after();
        const uint64_t va = sdesc_advance(vdesc, (Lv % C::SLOTS) * C::KV_TILE);
        if (leader) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            mma_ts(tmem + C::COL_O, tmem + C::COL_S + (T_ & 1) * BN + kk * 8,
                   sdesc_advance(va, kk * 16 * 128), idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
          // o_ready completes per key tile (waited only before a rescale of
          // O), o_done once per item.
          mma_commit(&bars->o_ready);
          if (j + 1 == n) mma_commit(&bars->o_done);
          mma_commit(&bars->ring_empty[Lv % C::SLOTS]);
        }
        if (j + 2 < n) {
          if (!(ok = wait_slot(loads + 2 * (j + 2)))) break;
          issue_s(T_ + 2, loads + 2 * (j + 2));
        }
      }
      loads += 2 * n;
      gt += n;
      ++q_cnt;
      ++items;
    }
    // Drain: all issued MMAs complete before TMEM is released.
    commit(&bars->drain);
    wait(&bars->drain, 0);
  } else {
    // ------------------------------------------------- softmax + epilogue
    // One thread per TMEM lane (query row).  These warps also move each Q
    // tile from its ring slots into TMEM, the next item's before the current
    // item's epilogue.
    const int quarter = warp & 3;  // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const float NEG_INF = __int_as_float(0xff800000);
    const float s_mul = CAP ? p.scale / p.softcap : p.scale * kLog2e;
    const float cap_mul = p.softcap * kLog2e;
    const bool up = p.scale > 0.0f;  // direction of the (monotone) score transform
    uint32_t gt = 0, taken = 0, done = 0;  // done: items with key tiles
    uint32_t lq = 0;  // ring loads accounted for (the producer's order)
    bool ok = true, q_pre = false;  // q_pre: the next item's Q is in TMEM
    T* out = static_cast<T*>(p.out);
    const int rows = G * m_tok;  // rows of the Q tile the TMA unit writes
    // Copies the next Q tile from its ring slots into TMEM (rows beyond the
    // tile as zeros) and signals the MMA warp.  Every S MMA of the previous
    // item has completed: its last S tile was waited for.
    auto copy_q = [&]() -> bool {
      bool got = true;
      for (int qs = 0; qs < C::Q_SLOTS; ++qs) {
        const uint32_t L = lq + qs;
        got = got && mbar_wait<false>(&bars->ring_full[L % C::SLOTS], (L / C::SLOTS) & 1, abort,
                                      status);
      }
      if (!__all_sync(0xffffffffu, got)) return false;
#pragma unroll 1
      for (int c = 0; c < C::KCH; ++c) {
        const uint32_t L = lq + c / C::Q_PER_SLOT;
        const uint8_t* src = smem + C::OFF_RING + (L % C::SLOTS) * C::KV_TILE +
                             (c % C::Q_PER_SLOT) * C::Q_CHUNK + r * 128;
        uint32_t w[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {  // 16-byte unit u of the row, 128-byte swizzle
          uint4 x = make_uint4(0, 0, 0, 0);
          if (r < rows) x = *reinterpret_cast<const uint4*>(src + ((u ^ (r & 7)) << 4));
          w[4 * u] = x.x;
          w[4 * u + 1] = x.y;
          w[4 * u + 2] = x.z;
          w[4 * u + 3] = x.w;
        }
        if (DQK % 64 == 0 || c + 1 < C::KCH) {
          tmem_st32(t_lane + C::COL_Q + c * 32, w);
        } else {  // a 32-column tail chunk
          uint32_t w16[16];
#pragma unroll
          for (int e = 0; e < 16; ++e) w16[e] = w[e];
          tmem_st16(t_lane + C::COL_Q + c * 32, w16);
        }
      }
      tmem_wait_st();
      fence_proxy_async_smem();  // the slots are refilled by the TMA unit next
      tc_fence_before();
      mbar_arrive(&bars->q_tmem);
      lq += C::Q_SLOTS;
      return true;
    };

    while (ok) {
      const int isl = taken % kItemSlots;
      ok = __all_sync(0xffffffffu, mbar_wait<false>(&bars->item_full[isl], (taken / kItemSlots) & 1,
                                             abort, status));
      if (!ok) break;
      const ItemSlot it = bars->items[isl];
      __syncwarp();
      if (lane == 0) mbar_arrive(&bars->item_empty[isl]);
      ++taken;
      if (it.last) break;
      const int n = it.n_tiles;
      const int tok = it.q0 + r / G;  // packed token of this row
      const int i = tok - it.q_start;  // its local query position
      const int first = it.t * m_tok;
      const bool own = r < G * m_tok && i >= first && i < min(first + m_tok, it.lq);
      const size_t orow = ((size_t)tok * p.H + (size_t)it.unit * G + (r % G)) * DV;
      if (n == 0) {
        if (own) {
#pragma unroll
          for (int c = 0; c < DV; c += 8)
            *reinterpret_cast<uint4*>(out + orow + c) = make_uint4(0, 0, 0, 0);
        }
        continue;
      }
      if (!q_pre && !(ok = copy_q())) break;
      q_pre = false;
      lq += 2 * n;
      const int off = it.lkv - it.lq;
      const int row_hi = p.is_causal ? min(it.lkv, i + off + 1) : it.lkv;
      const int row_lo = p.window > 0 ? i + off + 1 - p.window : 0;  // local window start
      float m_used = NEG_INF, l = 0.0f;

      for (int j = 0; j < n; ++j) {
        const uint32_t T_ = gt + j;
        ok = __all_sync(0xffffffffu,
                        mbar_wait<false>(&bars->s_full[T_ & 1], (T_ >> 1) & 1, abort, status));
        if (!ok) break;
        tc_fence_after();
        const uint32_t col_s = C::COL_S + (T_ & 1) * BN;
        uint32_t va[32], vb[32];
        tmem_ld32(t_lane + col_s, va);
        tmem_ld32(t_lane + col_s + 32, vb);
        tmem_wait_ld();
        const int J = it.jb + j;            // key tile index within the sequence
        const int k0 = min(it.kv_start + J * BN,
                           key_tile_limit(p, it.kv_start, it.lkv, total_kv) - BN);
        const int base = k0 - it.kv_start;  // local key index of column 0
        const int lo_c = max(J * BN, row_lo) - base;  // visible columns [lo_c, hi_c)
        const int hi_c = min((J + 1) * BN, row_hi) - base;
        const bool masked = !__all_sync(0xffffffffu, lo_c <= 0 && hi_c >= BN);
        uint32_t pw[32];
        float rs, alpha = 1.0f;
        {
          float mx, mn;
          if (masked)
            extremes64<true>(va, vb, lo_c, hi_c, mx, mn);
          else
            extremes64<false>(va, vb, lo_c, hi_c, mx, mn);
          const float ext = up ? mx : mn;  // the transform is monotone in the raw score
          const bool any = mx != NEG_INF;
          float mt = NEG_INF;
          if (any) mt = CAP ? cap_mul * tanh_via_exp2(ext * s_mul) : ext * s_mul;
          const float m_new = fmaxf(m_used, mt);
          if (m_new > m_used + kRescaleThreshold) {
            alpha = ex2_approx(m_used - m_new);  // 0 when m_used is -inf
            m_used = m_new;
          }
          const float m_eff = m_used == NEG_INF ? 0.0f : m_used;
          if (!CAP) {
            rs = masked ? exp64<T, 0, true>(va, vb, lo_c, hi_c, s_mul, cap_mul, m_eff, pw)
                        : exp64<T, 0, false>(va, vb, lo_c, hi_c, s_mul, cap_mul, m_eff, pw);
          } else {
            // every visible score of the warp has |t| <= 1/4: tanh from its series
            const float tmax = fmaxf(fabsf(mx * s_mul), fabsf(mn * s_mul));
            const bool series = __all_sync(0xffffffffu, !any || tmax <= kPolyLimit);
            if (series)
              rs = masked ? exp64<T, 1, true>(va, vb, lo_c, hi_c, s_mul, cap_mul, m_eff, pw)
                          : exp64<T, 1, false>(va, vb, lo_c, hi_c, s_mul, cap_mul, m_eff, pw);
            else
              rs = masked ? exp64<T, 2, true>(va, vb, lo_c, hi_c, s_mul, cap_mul, m_eff, pw)
                          : exp64<T, 2, false>(va, vb, lo_c, hi_c, s_mul, cap_mul, m_eff, pw);
          }
        }
        // P (16-bit pairs) over the S buffer's first 32 columns
        tmem_st32(t_lane + col_s, pw);
        l = l * alpha + rs;
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
          // O must hold PV(j-1) before it is rescaled.  S(j) was issued after
          // PV(j-2), so at most PV(j-1) is outstanding and the parity of its
          // phase is unambiguous.  P.V(j) itself needs no wait: it reads the
          // other S buffer and its MMAs follow P.V(j-1) in issue order.
          ok = __all_sync(0xffffffffu, mbar_wait<false>(&bars->o_ready, (T_ - 1) & 1, abort, status));
          if (!ok) break;
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < DV; c += 32) {
            uint32_t v[32];
            tmem_ld32(t_lane + C::COL_O + c, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
            tmem_st32(t_lane + C::COL_O + c, v);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(&bars->p_full[T_ & 1]);
      }
      if (!ok) break;

      // The next item's Q goes to TMEM before this item's epilogue, so that
      // its first S MMAs run meanwhile.
      {
        const int nsl = taken % kItemSlots;
        ok = __all_sync(0xffffffffu, mbar_wait<false>(&bars->item_full[nsl],
                                                      (taken / kItemSlots) & 1, abort, status));
        if (!ok) break;
        const ItemSlot nx = bars->items[nsl];
        if (!nx.last && nx.n_tiles > 0) {
          if (!(ok = copy_q())) break;
          q_pre = true;
        }
      }

      // epilogue: O / l -> out (rows of this item only).  When G divides 32
      // and every row of the warp belongs to this item, the warp's 32 rows
      // (32 / G whole tokens) leave through its 4 KB of staging and one
      // tensor store per 64 columns; otherwise each thread stores its row.
      ok = __all_sync(0xffffffffu, mbar_wait<false>(&bars->o_done, done & 1, abort, status));
      ++done;
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      const int own_lo = it.q_start + first, own_hi = it.q_start + min(first + m_tok, it.lq);
      const int tok_w = it.q0 + quarter * (32 / G);
      const bool staged =
          C::STAGE_BYTES > 0 && 32 % G == 0 && tok_w >= own_lo && tok_w + 32 / G <= own_hi;
      uint8_t* region = smem + C::OFF_STAGE + quarter * 4096;
#pragma unroll 1
      for (int c = 0; c < DV; c += 32) {
        uint32_t v[32];
        tmem_ld32(t_lane + C::COL_O + c, v);
        tmem_wait_ld();
        if (staged) {
          const bool lo_half = (c & 63) == 0;
          const int unit0 = lo_half ? 0 : 4;  // 16-byte units of the 128-byte row
          if (lo_half) {  // the region is free once the previous store has read it
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = 8 * u;
            uint4 w;
            w.x = pack2<T>(__uint_as_float(v[e + 0]) * inv, __uint_as_float(v[e + 1]) * inv);
            w.y = pack2<T>(__uint_as_float(v[e + 2]) * inv, __uint_as_float(v[e + 3]) * inv);
            w.z = pack2<T>(__uint_as_float(v[e + 4]) * inv, __uint_as_float(v[e + 5]) * inv);
            w.w = pack2<T>(__uint_as_float(v[e + 6]) * inv, __uint_as_float(v[e + 7]) * inv);
            *reinterpret_cast<uint4*>(region + lane * 128 + (((unit0 + u) ^ (lane & 7)) << 4)) = w;
          }
          if (!lo_half || c + 32 >= DV) {  // the 64-column box is complete (or the last)
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&tmap_o, region, c & ~63, it.unit * G, tok_w);
              bulk_commit();
            }
          }
        } else if (own) {
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
    }
    // Output stores must be complete before the CTA's shared memory goes.
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<C::TMEM_COLS>(tmem);
}

template <typename T, int DQK, int DV, bool CAP>
cudaError_t launch_tc(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                      const CUtensorMap& tv, const CUtensorMap& to, int num_sms, cudaStream_t s) {
  constexpr int smem = TcCfg<DQK, DV>::SMEM;
  auto kern = pva_prefill_tc_kernel<T, DQK, DV, CAP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, dim3(num_sms), dim3(kThreads), smem, s, p, tq, tk, tv, to);
}

template <typename T, int DQK, int DV>
cudaError_t launch_tc_cap(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                          const CUtensorMap& tv, const CUtensorMap& to, int num_sms,
                          cudaStream_t s) {
  return p.softcap != 0.0f ? launch_tc<T, DQK, DV, true>(p, tq, tk, tv, to, num_sms, s)
                           : launch_tc<T, DQK, DV, false>(p, tq, tk, tv, to, num_sms, s);
}

template <typename T>
cudaError_t launch_tc_shape(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& to, int num_sms,
                            cudaStream_t s) {
  if (p.d == 256 && p.dv == 256) return launch_tc_cap<T, 256, 256>(p, tq, tk, tv, to, num_sms, s);
  if (p.d == 192 && p.dv == 192) return launch_tc_cap<T, 192, 192>(p, tq, tk, tv, to, num_sms, s);
  if (p.d == 192 && p.dv == 128) return launch_tc_cap<T, 192, 128>(p, tq, tk, tv, to, num_sms, s);
  if (p.d == 96 && p.dv == 96) return launch_tc_cap<T, 96, 96>(p, tq, tk, tv, to, num_sms, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill_tc(const AttnParams& p, int dtype, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, int num_sms, cudaStream_t s) {
  return dtype == PVA_BF16 ? launch_tc_shape<__nv_bfloat16>(p, tq, tk, tv, to, num_sms, s)
                           : launch_tc_shape<__half>(p, tq, tk, tv, to, num_sms, s);
}

}  // namespace pva
