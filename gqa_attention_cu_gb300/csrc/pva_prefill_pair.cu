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
//   warp 0      TMA producer.  Decodes each work item once and publishes it
//               to the other roles through a small shared-memory ring, then
//               loads the item's two Q tiles and K_j, V_j into a ring of slots
//               (K and V separately, so K_{j+1} can land while V_j is read).
//   warp 1      MMA issuer + TMEM owner.  Order per key tile j:
//               PV0(j), S0(j+1), PV1(j), S1(j+1)  (S0(0), S1(0) up front).
//   warps 2..5  softmax / correction / epilogue for query tile 0
//   warps 6..9  the same for query tile 1
// TMEM (512 columns): S0 [0,128), S1 [128,256), O0 [256,256+d), O1 after O0.
// P_t (16-bit, two per column) overwrites the first 64 columns of S_t once
// they have been read, and the P.V MMA takes its A operand from TMEM; the
// next S_t MMA is issued after that P.V MMA (tcgen05 MMAs of one thread run in
// issue order).  Shared memory: Q0, Q1 (32 KB each at d = 128), a ring of
// K/V slots (4 of 32 KB at d = 128, 10 of 16 KB at d = 64) and two 16 KB
// output staging buffers.
//
// The softmax loops are specialised so that no uniform decision is taken per
// element: softcap on/off is a template parameter, and "tile needs a mask" and
// the sign of the scale are decided once per tile.  Pass 1 takes the row
// extreme of the raw scores with three-input max/min; pass 2 forms
// x*scale*log2(e) - m with packed fp32x2 FMAs, exponentiates with ex2 and
// sums with packed adds.
#include "pva_device.cuh"
#include "pva_items.cuh"
#include "pva_softmax.cuh"

namespace pva {
namespace {

constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;
constexpr int kMaxSlots = 12;
constexpr int kItemSlots = 4;
constexpr int kSoftmaxWarps = 8;

template <int D>
struct PairCfg {
  static constexpr int BN = 128;
  static constexpr int KCH = D / 64;
  static constexpr int Q_CHUNK = kTcRows * 128;       // 16 KB
  static constexpr int Q_TILE = KCH * Q_CHUNK;
  static constexpr int KV_CHUNK = BN * 128;           // 16 KB
  static constexpr int KV_TILE = KCH * KV_CHUNK;
  static constexpr int SLOTS = D == 128 ? 4 : 10;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = 2 * Q_TILE;
  static constexpr int STAGE = kTcRows * 128;                // 64 output columns of a tile
  static constexpr int OFF_STAGE = OFF_RING + SLOTS * KV_TILE;  // one buffer per query tile
  static constexpr int OFF_BAR = OFF_STAGE + 2 * STAGE;
  static constexpr int SMEM = OFF_BAR + 1024 + 1024;  // barriers/item ring + alignment slack
  static constexpr int TMEM_COLS = 512;
  static constexpr int COL_S = 0;        // + 128 * tile
  static constexpr int COL_O = 256;      // + D * tile
  static_assert(SLOTS <= kMaxSlots, "barrier array");
  static_assert(2 * BN + 2 * D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM <= 232448 - 64, "shared memory budget");
};

// A decoded work item, as the producer publishes it.
struct ItemSlot {
  int q_start, kv_start, lq, lkv;
  int t, unit, n_tiles, q0;
  int last;  // 1: no more items for this CTA
  int jb;  // first key tile (a local window skips the ones before)
  int empty;  // bit t: query tile t owns no row of the item
  int pad;
};

struct PairBars {
  uint64_t q_full, q_empty, drain, pad;
  uint64_t s_full[2], p_half[2], p_full[2], o_ready[2], o_free[2];
  uint64_t stage_full[2], stage_free[2];  // epilogue staging buffer hand-off
  uint64_t ring_full[kMaxSlots], ring_empty[kMaxSlots];
  uint64_t item_full[kItemSlots], item_empty[kItemSlots];
  ItemSlot items[kItemSlots];
};
static_assert(sizeof(PairBars) <= 1024, "barrier block");

template <typename T, int D, bool CAP, bool UP>
__global__ void __launch_bounds__(kThreads, 1)
    pva_prefill_pair_kernel(AttnParams p, const __grid_constant__ CUtensorMap tmap_q,
                            const __grid_constant__ CUtensorMap tmap_k,
                            const __grid_constant__ CUtensorMap tmap_v,
                            const __grid_constant__ CUtensorMap tmap_o) {
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
  const int total_kv = kv_tile_end(p);

  if (threadIdx.x == 0) {
    s_abort = 0;
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    mbar_init(&bars->drain, 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_half[t], 128);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_ready[t], 1);
      mbar_init(&bars->o_free[t], 128);
      mbar_init(&bars->stage_full[t], 128);
      mbar_init(&bars->stage_free[t], 1);
    }
    for (int s = 0; s < C::SLOTS; ++s) {
      mbar_init(&bars->ring_full[s], 1);
      mbar_init(&bars->ring_empty[s], 1);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      mbar_init(&bars->item_full[s], 1);
      mbar_init(&bars->item_empty[s], 1 + kSoftmaxWarps);  // MMA thread + one lane per warp
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
    prefetch_tensor_map(&tmap_o);
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
      uint32_t items = 0, loads = 0, published = 0;
      const uint32_t q_bytes = 2u * C::KCH * (uint32_t)(G * m_tok) * 128u;
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
      // next item is decoded (a few dependent reads of the scheduler's lists)
      // once the current item's first loads are out, so both latencies
      // overlap the current item instead of delaying the next publish.
      int* next_item = p.ws + WsLayout{p.B, p.Hkv}.counters();
      int idx = atomicAdd(next_item, 1);
      PrefillItem it{};
      if (idx < h.n_items) it = decode_prefill_item(p, h, idx);
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
        v.q0 = min(it.q_start + it.t * h.tile_tokens, total_q - 2 * m_tok);
        v.last = 0;
        v.empty = 0;
        {
          const int first = it.t * h.tile_tokens, lo0 = v.q0 - it.q_start;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int a = max(first, lo0 + t * m_tok);
            const int b = min(min(first + h.tile_tokens, it.lq), lo0 + (t + 1) * m_tok);
            if (a >= b) v.empty |= 1 << t;
          }
        }
        if (!(ok = publish(v))) break;
        if (v.n_tiles > 0) {
          const int g = v.unit;
          if (!(ok = mbar_wait<false>(&bars->q_empty, (items & 1) ^ 1, abort, status))) break;
          mbar_arrive_expect_tx(&bars->q_full, q_bytes);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_load_3d(smem + C::OFF_Q + t * C::Q_TILE + c * C::Q_CHUNK, &tmap_q,
                          &bars->q_full, c * 64, g * G, v.q0 + t * m_tok);
          ++items;
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
              mbar_arrive_expect_tx(&bars->ring_full[sl], (uint32_t)C::KV_TILE);
#pragma unroll
              for (int c = 0; c < C::KCH; ++c)
                load_kv_box(dst + c * C::KV_CHUNK, kv ? &tmap_v : &tmap_k, &bars->ring_full[sl], p,
                            c * 64, it.b, g, v.kv_start, k0);
            }
            if (!decoded) {
              it_next = decode_prefill_item(p, h, idx_next);
              decoded = true;
            }
          }
        }
        if (!ok) break;
        if (!decoded) it_next = decode_prefill_item(p, h, idx_next);
        idx = idx_next;
        it = it_next;
      }
      if (ok) {
        ItemSlot v{};
        v.last = 1;
        publish(v);
      }
      // Drain: every copy this thread issued must land before the CTA exits.
      if (items) mbar_wait<false>(&bars->q_full, (items - 1) & 1, abort, status);
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
    constexpr uint32_t idesc_o = idesc_f16<T>(kTcRows, D, false, true);
    // Base descriptors, built once: the issue loops only add constants.
    const uint64_t qdesc = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
    const uint64_t kdesc = sdesc_sw128(smem_u32(smem + C::OFF_RING), 16, 1024);
    const uint64_t vdesc = sdesc_sw128(smem_u32(smem + C::OFF_RING), C::KV_CHUNK, 1024);
    uint32_t items = 0, loads = 0, tiles = 0, taken = 0;
    bool ok = true;
    auto commit = [&](uint64_t* bar) {
      if (leader) mma_commit(bar);
    };
    int empty = 0;  // bit t: query tile t of the current item owns no row
    auto issue_s = [&](int t, uint32_t kslot) {
      const uint64_t qa = sdesc_advance(qdesc, t * C::Q_TILE);
      const uint64_t ka = sdesc_advance(kdesc, kslot * C::KV_TILE);
      if (leader) {
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          if ((empty >> t) & 1) break;
          const uint32_t off = (kk & 3) * 32;
          mma_ss(tmem + C::COL_S + t * 128, sdesc_advance(qa, (kk >> 2) * C::Q_CHUNK + off),
                 sdesc_advance(ka, (kk >> 2) * C::KV_CHUNK + off), idesc_s, kk > 0 ? 1u : 0u);
        }
        mma_commit(&bars->s_full[t]);
      }
    };
    // P.V for keys [16 k0, 16 k1) of the tile (P columns 8 k0 .. 8 k1)
    auto issue_pv = [&](int t, uint32_t vslot, bool first, int k0, int k1) {
      const uint64_t va = sdesc_advance(vdesc, vslot * C::KV_TILE);
      if (leader) {
#pragma unroll
        for (int kk = k0; kk < k1; ++kk) {
          if ((empty >> t) & 1) break;
          mma_ts(tmem + C::COL_O + t * D, tmem + C::COL_S + t * 128 + kk * 8,
                 sdesc_advance(va, kk * 16 * 128), idesc_o, (!first || kk > 0) ? 1u : 0u);
        }
        if (k1 == BN / 16) mma_commit(&bars->o_ready[t]);
      }
    };
    auto wait = [&](uint64_t* bar, uint32_t parity) -> bool {
      return __all_sync(0xffffffffu, mbar_wait<false>(bar, parity, abort, status));
    };
    auto wait_slot = [&](uint32_t L) -> bool {
      const bool r = wait(&bars->ring_full[L % C::SLOTS], (L / C::SLOTS) & 1);
      tc_fence_after();
      return r;
    };
    // P.V of tile t in two halves, each after its half of P has been written
    auto pv_halves = [&](int t, uint32_t vslot, bool first, uint32_t T_) -> bool {
      if (!wait(&bars->p_half[t], T_ & 1)) return false;
      tc_fence_after();
      issue_pv(t, vslot, first, 0, BN / 32);
      if (!wait(&bars->p_full[t], T_ & 1)) return false;
      tc_fence_after();
      issue_pv(t, vslot, first, BN / 32, BN / 16);
      return true;
    };
    while (ok) {
      const int isl = taken % kItemSlots;
      if (!(ok = wait(&bars->item_full[isl], (taken / kItemSlots) & 1))) break;
      const int n = bars->items[isl].n_tiles, last = bars->items[isl].last;
      empty = bars->items[isl].empty;
      __syncwarp();
      if (leader) mbar_arrive(&bars->item_empty[isl]);
      ++taken;
      if (last) break;
      if (n == 0) continue;
      if (!(ok = wait(&bars->q_full, items & 1))) break;
      tc_fence_after();
      // key tile j lives in load slots (loads + 2j) (K) and (loads + 2j + 1) (V)
      if (!(ok = wait_slot(loads))) break;
      issue_s(0, loads % C::SLOTS);
      issue_s(1, loads % C::SLOTS);
      commit(&bars->ring_empty[loads % C::SLOTS]);
      if (n == 1) commit(&bars->q_empty);
      for (int j = 0; ok && j < n; ++j) {
        const uint32_t Lk = loads + 2 * j, Lv = Lk + 1, Lk1 = Lk + 2;
        const uint32_t T_ = tiles + j;
        // V_j and K_{j+1} have normally landed long before P0(j) is ready:
        // wait for them first, so that nothing but the issue itself follows
        // the P0(j) arrival.
        if (!(ok = wait_slot(Lv))) break;
        if (j + 1 < n && !(ok = wait_slot(Lk1))) break;
        // PV0(j)
        if (j == 0 && !(ok = wait(&bars->o_free[0], (items & 1) ^ 1))) break;
        if (!(ok = pv_halves(0, Lv % C::SLOTS, j == 0, T_))) break;
        // S0(j+1)
        if (j + 1 < n) issue_s(0, Lk1 % C::SLOTS);
        // PV1(j)
        if (j == 0 && !(ok = wait(&bars->o_free[1], (items & 1) ^ 1))) break;
        if (!(ok = pv_halves(1, Lv % C::SLOTS, j == 0, T_))) break;
        commit(&bars->ring_empty[Lv % C::SLOTS]);
        // S1(j+1)
        if (j + 1 < n) {
          issue_s(1, Lk1 % C::SLOTS);
          commit(&bars->ring_empty[Lk1 % C::SLOTS]);
          if (j + 2 == n) commit(&bars->q_empty);
        }
      }
      loads += 2 * n;
      tiles += n;
      ++items;
    }
    // Drain: all issued MMAs complete before TMEM is released.
    commit(&bars->drain);
    wait(&bars->drain, 0);
  } else {
    // ------------------------------------------------- softmax + epilogue
    const int tq = warp >= 6 ? 1 : 0;  // query tile of this warpgroup
    const int quarter = warp & 3;      // TMEM lanes this warp may access
    const int r = quarter * 32 + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t col_s = C::COL_S + tq * 128, col_o = C::COL_O + tq * D;
    const float NEG_INF = __int_as_float(0xff800000);
    const float s_mul = CAP ? p.scale / p.softcap : p.scale * kLog2e;
    const float cap_mul = p.softcap * kLog2e;
    const int span = 2 * m_tok;      // tokens per item
    uint32_t tiles = 0, taken = 0, stages = 0;
    bool ok = true;
    T* out = static_cast<T*>(p.out);

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
      const int tok = it.q0 + tq * m_tok + r / G;
      const int i = tok - it.q_start;
      const int first = it.t * span;
      const bool own = r < G * m_tok && i >= first && i < min(first + span, it.lq);
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
      const int row_lo = p.window > 0 ? i + off + 1 - p.window : 0;  // local window start
      float m_used = NEG_INF, l = 0.0f;

      for (int j = 0; j < n; ++j) {
        const uint32_t T_ = tiles + j;
        ok = __all_sync(0xffffffffu, mbar_wait<false>(&bars->s_full[tq], T_ & 1, abort, status));
        if (!ok) break;
        tc_fence_after();
        if ((it.empty >> tq) & 1) {  // no row of this tile is owned: no P, no P.V
          mbar_arrive(&bars->p_half[tq]);
          mbar_arrive(&bars->p_full[tq]);
          continue;
        }
        const int J = it.jb + j;            // key tile index within the sequence
        const int k0 = min(it.kv_start + J * BN,
                           key_tile_limit(p, it.kv_start, it.lkv, total_kv) - BN);
        const int base = k0 - it.kv_start;  // local key index of column 0
        const int lo_c = max(J * BN, row_lo) - base;  // visible columns [lo_c, hi_c)
        const int hi_c = min((J + 1) * BN, row_hi) - base;
        // Per 64-column half, decided once for the warp: every column visible,
        // a one-sided mask (no row starts inside the half), a two-sided mask,
        // or nothing visible (the half is skipped: P = 0, no exponentials).
        int mode[BN / 64];
#pragma unroll
        for (int c = 0; c < BN; c += 64) {
          mode[c / 64] = __all_sync(0xffffffffu, lo_c <= c && hi_c >= c + 64) ? kMaskNone
                         : __all_sync(0xffffffffu, hi_c <= c || lo_c >= c + 64 || hi_c <= lo_c)
                             ? kHalfEmpty
                         : __all_sync(0xffffffffu, lo_c <= c) ? kMaskHi
                                                               : kMaskBoth;
        }
        // Pass 1: extreme raw score over the visible columns.  The score
        // transform (scale, then optional softcap) is monotone -- increasing
        // for scale > 0, decreasing for scale < 0 -- so the row max of the
        // transformed scores is the transform of this extreme.
        float ext = UP ? NEG_INF : -NEG_INF;
#pragma unroll
        for (int c = 0; c < BN; c += 64) {
          const int md = mode[c / 64];
          if (md == kHalfEmpty) continue;
          uint32_t va[32], vb[32];
          tmem_ld32(t_lane + col_s + c, va);
          tmem_ld32(t_lane + col_s + c + 32, vb);
          tmem_wait_ld();
          ext = md == kMaskNone ? extreme64<UP, kMaskNone>(va, vb, c, lo_c, hi_c, ext)
                : md == kMaskHi ? extreme64<UP, kMaskHi>(va, vb, c, lo_c, hi_c, ext)
                                : extreme64<UP, kMaskBoth>(va, vb, c, lo_c, hi_c, ext);
        }
        const float mt = (ext == NEG_INF || ext == -NEG_INF)
                             ? NEG_INF
                             : (CAP ? cap_mul * tanh_via_exp2(ext * s_mul) : ext * s_mul);
        const float m_new = fmaxf(m_used, mt);
        float alpha = 1.0f;
        if (m_new > m_used + kRescaleThreshold) {
          alpha = ex2_approx(m_used - m_new);  // 0 when m_used is -inf
          m_used = m_new;
        }
        const float m_eff = m_used == NEG_INF ? 0.0f : m_used;
        // O holds the P.V products of tiles < j: the P.V MMA of tile j-1 was
        // issued before the S MMA of tile j, and tcgen05 operations of one
        // thread complete in order, so the s_full arrival above already
        // covers it.
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.0f)) {
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
        // Pass 2: p = 2^(x - m), row sum, P (16-bit pairs) into TMEM over the
        // S columns already read: columns [c, c+64) of S become P columns
        // [c/2, c/2 + 32).
        float2 rs = make_float2(0.0f, 0.0f);
#pragma unroll
        for (int c = 0; c < BN; c += 64) {
          const int md = mode[c / 64];
          uint32_t pw[32];
          if (md == kHalfEmpty) {
#pragma unroll
            for (int e = 0; e < 32; ++e) pw[e] = 0u;
          } else {
            uint32_t va[32], vb[32];
            tmem_ld32(t_lane + col_s + c, va);
            tmem_ld32(t_lane + col_s + c + 32, vb);
            tmem_wait_ld();
            if (md == kMaskNone)
              exp64<T, CAP, kMaskNone>(va, vb, c, lo_c, hi_c, s_mul, cap_mul, m_eff, rs, pw);
            else if (md == kMaskHi)
              exp64<T, CAP, kMaskHi>(va, vb, c, lo_c, hi_c, s_mul, cap_mul, m_eff, rs, pw);
            else
              exp64<T, CAP, kMaskBoth>(va, vb, c, lo_c, hi_c, s_mul, cap_mul, m_eff, rs, pw);
          }
          tmem_st32(t_lane + col_s + (c >> 1), pw);
          tmem_wait_st();
          tc_fence_before();
          // The first half of P lets the P.V MMA start on keys [0, 64)
          // while the second half is computed.
          mbar_arrive(c == 0 ? &bars->p_half[tq] : &bars->p_full[tq]);
        }
        l = l * alpha + (rs.x + rs.y);
      }
      if (!ok) break;

      // epilogue: O / l -> out (rows of this item only)
      const uint32_t T_last = tiles + n - 1;
      ok = __all_sync(0xffffffffu, mbar_wait<false>(&bars->o_ready[tq], T_last & 1, abort, status));
      if (!ok) break;
      tc_fence_after();
      const float inv = l > 0.0f ? 1.0f / l : 0.0f;
      // A tile whose m tokens all belong to this item goes out through shared
      // memory and one TMA store per 64 columns; otherwise (the last tile of
      // a sequence) each thread stores its own row.
      const int tok0 = it.q0 + tq * m_tok;
      const int own_lo = it.q_start + first, own_hi = it.q_start + min(first + span, it.lq);
      const bool whole = tok0 >= own_lo && tok0 + m_tok <= own_hi;
      uint8_t* stage = smem + C::OFF_STAGE + tq * C::STAGE;
      const bool issuer = r == 0;  // lane 0 of the warp with lane quarter 0
      // G dividing 32: each warp's rows are whole tokens and go out on their own.
      const bool per_warp = 32 % G == 0;
      const int tok_w = tok0 + quarter * (32 / G);
      const bool warp_whole = tok_w >= own_lo && tok_w + 32 / G <= own_hi;
      // 32 columns at a time; a TMA store leaves per 64-column half.
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        const bool first = (c & 63) == 0, second = !first;  // position within the half
        const int unit0 = second ? 4 : 0;                    // 16-byte units of the 128-byte row
        uint32_t w[16];  // the row's 32 values of columns [c, c + 32), packed
        {
          uint32_t v[32];
          tmem_ld32(t_lane + col_o + c, v);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; e += 2)
            w[e >> 1] = pack2<T>(__uint_as_float(v[e]) * inv, __uint_as_float(v[e + 1]) * inv);
        }
        if (per_warp) {
          // This warp's 32 rows (32 / G whole tokens) leave in their own
          // 4 KB box: no barrier across the warpgroup.  Lane 0 first waits
          // until its previous store has read the region.
          if (warp_whole) {
            uint8_t* region = stage + quarter * (32 * 128);
            if (first) {
              if (lane == 0) bulk_wait_read_all();
              __syncwarp();
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(region + lane * 128 + (((unit0 + u) ^ (lane & 7)) << 4)) =
                  make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
            if (second) {
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&tmap_o, region, c - 32, it.unit * G, tok_w);
                bulk_commit();
              }
            }
          } else if (own) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(out + orow + c + 8 * u) =
                  make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          }
        } else if (whole) {
          if (first) {
            // The staging buffer is free once the previous store has read it.
            if (issuer) {
              bulk_wait_read_all();
              mbar_arrive(&bars->stage_free[tq]);
            }
            ok = __all_sync(0xffffffffu,
                            mbar_wait<false>(&bars->stage_free[tq], stages & 1, abort, status));
            if (!ok) break;
          }
          // Row r: 128 bytes in the 128-byte swizzled layout of the TMA box.
          if (r < G * m_tok) {
#pragma unroll
            for (int u = 0; u < 4; ++u)
              *reinterpret_cast<uint4*>(stage + r * 128 + (((unit0 + u) ^ (r & 7)) << 4)) =
                  make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
          }
          if (second) {
            fence_proxy_async_smem();
            mbar_arrive(&bars->stage_full[tq]);
            if (issuer) {
              if (!(ok = mbar_wait<false>(&bars->stage_full[tq], stages & 1, abort, status))) break;
              tma_store_3d(&tmap_o, stage, c - 32, it.unit * G, tok0);
              bulk_commit();
            }
            ++stages;
          }
        } else if (own) {
#pragma unroll
          for (int u = 0; u < 4; ++u)
            *reinterpret_cast<uint4*>(out + orow + c + 8 * u) =
                make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
      if (!ok) break;
      tc_fence_before();
      mbar_arrive(&bars->o_free[tq]);
      tiles += n;
    }
    // Output stores must be complete before the CTA's shared memory goes.
    if (lane == 0) bulk_wait_all();
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc<C::TMEM_COLS>(tmem);
}

template <typename T, int D, bool CAP, bool UP>
cudaError_t launch_pair(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, const CUtensorMap& to, int num_sms,
                        cudaStream_t s) {
  constexpr int smem = PairCfg<D>::SMEM;
  auto kern = pva_prefill_pair_kernel<T, D, CAP, UP>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, dim3(num_sms), dim3(kThreads), smem, s, p, tq, tk, tv, to);
}

template <typename T, int D>
cudaError_t launch_pair_cap(const AttnParams& p, const CUtensorMap& tq, const CUtensorMap& tk,
                            const CUtensorMap& tv, const CUtensorMap& to, int num_sms,
                            cudaStream_t s) {
  // UP: direction of the (monotone) score transform, from the sign of the scale
  if (p.scale > 0.0f)
    return p.softcap != 0.0f ? launch_pair<T, D, true, true>(p, tq, tk, tv, to, num_sms, s)
                             : launch_pair<T, D, false, true>(p, tq, tk, tv, to, num_sms, s);
  return p.softcap != 0.0f ? launch_pair<T, D, true, false>(p, tq, tk, tv, to, num_sms, s)
                           : launch_pair<T, D, false, false>(p, tq, tk, tv, to, num_sms, s);
}

}  // namespace

cudaError_t launch_prefill_pair(const AttnParams& p, int dtype, const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, int num_sms, cudaStream_t s) {
  const bool bf = dtype == PVA_BF16;
  switch (p.d) {
    case 64:
      return bf ? launch_pair_cap<__nv_bfloat16, 64>(p, tq, tk, tv, to, num_sms, s)
                : launch_pair_cap<__half, 64>(p, tq, tk, tv, to, num_sms, s);
    case 128:
      return bf ? launch_pair_cap<__nv_bfloat16, 128>(p, tq, tk, tv, to, num_sms, s)
                : launch_pair_cap<__half, 128>(p, tq, tk, tv, to, num_sms, s);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pva
