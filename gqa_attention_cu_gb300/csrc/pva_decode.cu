// Split-KV decode for sequences with a single query token (L_q == 1), bf16 or
// f16, head sizes (d, dv) in {(64,64), (96,96), (128,128), (192,192),
// (256,256), (192,128)}, H/Hkv = G in {1, 2, 4, 8, 16}.
//
// With one query row the tail-aligned causal frontier (packed_varlen_
// attention.rs, "Causal alignment") is L_kv - 1, so every key is visible and
// the work is a pass over the sequence's K and V rows: it is bound by HBM
// bandwidth, and each K/V row is read once for all G query heads that share
// it.
//
// Work unit = (sequence, kv head g, split s): the keys of a sequence are cut
// into S_b splits (chosen on the device by the scheduler).  Per CTA
// (persistent, one per SM):
//   warp 0      TMA producer: draws units from a device-wide counter,
//               publishes each decoded unit through a shared-memory ring, and
//               streams its K and V tiles of TK keys (16 KB each, rows of d
//               contiguous elements) into a ring of up to 6 stages.
//   warps 1..NW compute (NW = 12 or 8 by head shape, see DecCfg).  A warp serves
//               GW = min(G, 8) heads at d = 64, min(G, 4) at larger head
//               sizes; with more heads than that the warps split into head
//               groups over the same tiles (G = 16, d = 128: warps 1..3 take
//               heads 0..3, warps 4..6 heads 4..7, and so on).  A round
//               covers R = 32/GW keys x GW heads = 32 (key, head) pairs:
//               lane l owns DPL consecutive dims of every key (DPL = 2, 4 or
//               8; lanes past the head size hold zeros), forms the 32
//               partial dot products, and a reduce-scatter butterfly (warp
//               shuffles) leaves the full score of pair l in lane l.  Online softmax
//               per head, probabilities shared through shared memory, O
//               accumulated per lane over its dims of V.  Rounds are dealt to
//               the warps across tiles, so with fewer rounds per tile than
//               warps (small G) each warp takes whole tiles in turn.
//   end of unit the NW warps' (max, sum, O) are merged in a fixed order;
//               an unsplit unit writes the output row; a split unit writes
//               its fp32 partial and the last split to finish (device-wide
//               counter) combines all splits in split order (log-sum-exp
//               combine) and writes the output, so results do not depend on
//               which CTA finishes last.
#include "pva_device.cuh"
#include "pva_items.cuh"

namespace pva {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kUnitSlots = 4;

// Dims per lane for a head size (the smallest of 2, 4, 8 that covers it
// with 32 lanes); lanes [D / DPL, 32) hold no dims.
__host__ __device__ constexpr int dims_per_lane(int D) { return D <= 64 ? 2 : D <= 128 ? 4 : 8; }

template <int DK, int DV, int G>
struct DecCfg {
  // Heads per warp: up to 8 at d = 64, else up to 4.  At head sizes >= 192
  // the per-lane q and O of 8 heads (8 dims each) spilled to local memory
  // (d = 256, G = 8: 2.0 ms -> 1.16 ms for 4.6 GB of K/V); at d = 96 and 128
  // 4 heads per warp keep a lane's arrays within the 128 registers of 12
  // compute warps, and G = 8 / 16 ran 6% / 4% faster that way (more, shorter
  // rounds, each K/V tile read from shared memory by 2 or 4 head groups)
  // than with 8 heads on 8 warps; at d = 64 8 heads per warp stayed 2%
  // faster.
  static constexpr int GW = DK > 64 ? (G < 4 ? G : 4) : (G < 8 ? G : 8);
  static constexpr int DPLK = dims_per_lane(DK), DPLV = dims_per_lane(DV);
  // Compute warps: 12 where a warp serves 4 or more heads (many short
  // rounds per tile) and a lane's q, O and 32 partial scores still fit the
  // 128 registers that 13 warps per SM leave each thread; else 8.  A round
  // is a long dependent chain (dot products, shuffle butterfly, softmax,
  // P.V), and with 3 compute warps per sub-partition instead of 2 more of
  // them overlap: d = 128, G = 4: 0.80 -> 0.76 ms (256 sequences); d = 64,
  // G = 4 / 8 / 16: 9-12% faster.  With 1 or 2 heads per warp a tile holds
  // few rounds and 12 warps gained nothing (d = 256, G = 1: 2% slower); the
  // wider head shapes spill at 12.
  static constexpr int NW =
      GW >= 4 && GW * (DPLK > DPLV ? DPLK : DPLV) <= (DK >= 192 ? 8 : 16) ? 12 : 8;
  static constexpr int THREADS = 32 * (1 + NW);
  static constexpr int HG = G / GW;                // head groups
  static constexpr int NWG = NW / HG;              // warps per head group
  static constexpr int TK = decode_tile_keys(DK, DV);  // keys per tile
  static constexpr int LK = DK / DPLK, LV = DV / DPLV;  // lanes holding dims
  static constexpr int R = 32 / GW;                // keys per round
  static constexpr int RPT = TK / R;               // rounds per tile
  static constexpr int K_BYTES = TK * DK * 2;
  static constexpr int V_BYTES = TK * DV * 2;
  static constexpr int STAGE = K_BYTES + V_BYTES;
  static constexpr int OFF_KV = 0;
  // K/V ring: as many 32 KB stages as shared memory holds next to the merge
  // buffers, at most 6 (6 at every shape built; 4 measured 1-5% slower:
  // bf16_decode 0.762 -> 0.756 ms, d = 128, G = 1 2.51 -> 2.44 ms).
  static constexpr int REST = NW * GW * DV * 4 + 2 * NW * GW * 4 + NW * 32 * 4 + NW * GW * 4 +
                              2 * 6 * 8 + 2 * kUnitSlots * 8 + kUnitSlots * 64 + 128;
  static constexpr int STAGES = (232448 - REST) / STAGE < 6 ? (232448 - REST) / STAGE : 6;
  static_assert(STAGES >= 4, "K/V ring depth");
  static constexpr int OFF_O = STAGES * STAGE;             // [NW][GW][DV] fp32
  static constexpr int OFF_ML = OFF_O + NW * GW * DV * 4;   // [NW][GW] m, [NW][GW] l
  static constexpr int OFF_P = OFF_ML + 2 * NW * GW * 4;    // [NW][32] p
  static constexpr int OFF_A = OFF_P + NW * 32 * 4;         // [NW][GW] alpha
  static constexpr int OFF_BAR = OFF_A + NW * GW * 4;
  static constexpr int OFF_UNITS = OFF_BAR + 2 * STAGES * 8 + 2 * kUnitSlots * 8;
  static constexpr int SMEM = OFF_UNITS + kUnitSlots * 64 + 128;
  static_assert(G % GW == 0 && NW % HG == 0, "head groups");
  static_assert(DK % DPLK == 0 && DV % DPLV == 0, "dims per lane");
  static_assert(RPT >= 1 && TK % R == 0, "tile shorter than a round");
  static_assert(K_BYTES % 128 == 0 && V_BYTES % 128 == 0, "tile alignment");
  static_assert(SMEM <= 232448, "shared memory budget");
};

struct Unit {
  int b, g, s, S;      // sequence, kv head, split index, split count
  int ks, ke;          // key range [ks, ke) local to the sequence
  int kv_start, q_tok;
  int u, last;         // unit index (partial slot); 1: no more units for this CTA
  int pad[6];
};
static_assert(sizeof(Unit) == 64, "unit slot");

__device__ __forceinline__ Unit decode_unit(const AttnParams& p, const SchedHeader& h, int u) {
  const WsLayout L{p.B, p.Hkv};
  const int32_t* order = p.ws + L.dec_order();
  const int32_t* prefix = p.ws + L.dec_prefix();
  int lo = 0, hi = h.n_dec - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
  }
  Unit r;
  r.b = order[lo];
  r.S = (prefix[lo + 1] - prefix[lo]) / p.Hkv;
  const int local = u - prefix[lo];
  r.g = local / r.S;
  r.s = local - r.g * r.S;
  r.kv_start = p.cu_kv[r.b];
  r.q_tok = p.cu_q[r.b];
  const int lkv = p.kv_len ? p.kv_len[r.b] : p.cu_kv[r.b + 1] - r.kv_start;
  // A local window W keeps the last W keys (the one query row sits at the end).
  const int kbeg = p.window > 0 && p.window < lkv ? lkv - p.window : 0;
  const int per = (lkv - kbeg + r.S - 1) / r.S;
  r.ks = min(lkv, kbeg + r.s * per);
  r.ke = min(lkv, r.ks + per);
  return r;
}

// First row (packed row index) of tile j of a unit.  Packed K/V: tiles are
// shifted back only at the end of the tensor (rows past the unit are other
// sequences' keys, weighted 0).  Cache planes and padded slots: the unit's
// last tile is shifted back to end at the unit's last key -- before row 0 of
// the plane or slot, where the tensor copy reads zeros, if the unit is shorter
// than a tile -- so no row past the sequence's keys, which holds whatever the
// cache or the padding held, is ever loaded.  The rows a shifted tile repeats
// are masked as already seen.
template <int TK>
__device__ __forceinline__ int tile_row(const AttnParams& p, const Unit& un, int j,
                                        int total_kv) {
  const int lim = p.kv_cap || p.kv_slot ? un.kv_start + un.ke : total_kv;
  return min(un.kv_start + un.ks + j * TK, lim - TK);
}

template <int NW>
__device__ __forceinline__ void compute_bar_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(NW * 32) : "memory");
}

template <typename T, int N>
__device__ __forceinline__ void load_dims(const uint8_t* row, int lane, float (&f)[N]) {
  // N consecutive 16-bit values at element offset lane * N.
  const uint8_t* src = row + lane * N * 2;
  if constexpr (N == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
    const float2 a = unpack2<T>(w);
    f[0] = a.x; f[1] = a.y;
  } else if constexpr (N == 4) {
    const uint2 w = *reinterpret_cast<const uint2*>(src);
    const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const float2 a = unpack2<T>(w.x), b = unpack2<T>(w.y), c = unpack2<T>(w.z),
                 d = unpack2<T>(w.w);
    f[0] = a.x; f[1] = a.y; f[2] = b.x; f[3] = b.y;
    f[4] = c.x; f[5] = c.y; f[6] = d.x; f[7] = d.y;
  }
}

// G consecutive probabilities of one key (a broadcast shared-memory read).
template <int G>
__device__ __forceinline__ void load_probs(const float* src, float (&p)[G]) {
  if constexpr (G >= 4) {
#pragma unroll
    for (int i = 0; i < G; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(src + i);
      p[i] = v.x; p[i + 1] = v.y; p[i + 2] = v.z; p[i + 3] = v.w;
    }
  } else if constexpr (G == 2) {
    const float2 v = *reinterpret_cast<const float2*>(src);
    p[0] = v.x; p[1] = v.y;
  } else {
    p[0] = src[0];
  }
}

template <typename T, int DK, int DV, int G>
__global__ void __launch_bounds__(DecCfg<DK, DV, G>::THREADS, 1)
    pva_decode_kernel(AttnParams p, const __grid_constant__ CUtensorMap tmap_k,
                      const __grid_constant__ CUtensorMap tmap_v) {
  using C = DecCfg<DK, DV, G>;
  constexpr int TK = C::TK, DPLK = C::DPLK, DPLV = C::DPLV, R = C::R, GW = C::GW;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                             ~uintptr_t(127));
  float* sO = reinterpret_cast<float*>(smem + C::OFF_O);
  float* sM = reinterpret_cast<float*>(smem + C::OFF_ML);
  float* sL = sM + C::NW * GW;
  float* sP = reinterpret_cast<float*>(smem + C::OFF_P);
  float* sA = reinterpret_cast<float*>(smem + C::OFF_A);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
  uint64_t* empty = full + C::STAGES;
  uint64_t* unit_full = empty + C::STAGES;
  uint64_t* unit_empty = unit_full + kUnitSlots;
  Unit* units = reinterpret_cast<Unit*>(smem + C::OFF_UNITS);
  __shared__ int s_abort, s_last;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  uint32_t* status = p.status;
  volatile int* abort = &s_abort;
  const int total_kv = kv_tile_end(p);

  if (threadIdx.x == 0) {
    s_abort = 0;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NW);
    }
    for (int s = 0; s < kUnitSlots; ++s) {
      mbar_init(&unit_full[s], 1);
      mbar_init(&unit_empty[s], C::NW);
    }
    fence_mbar_init();
  }
  __syncthreads();
  wait_prior_grid();  // the scheduler's work lists are complete from here on
  allow_next_grid();  // the prefill kernel may start its set-up
  const SchedHeader h = *reinterpret_cast<const SchedHeader*>(p.ws + kWsHeader);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tensor_map(&tmap_k);
      prefetch_tensor_map(&tmap_v);
      uint32_t cnt = 0, published = 0;
      bool ok = true;
      auto publish = [&](const Unit& v) -> bool {
        const int sl = published % kUnitSlots;
        if (!mbar_wait(&unit_empty[sl], ((published / kUnitSlots) & 1) ^ 1, abort, status))
          return false;
        units[sl] = v;
        mbar_arrive(&unit_full[sl]);
        ++published;
        return true;
      };
      // Units are drawn from a device-wide counter (zeroed by the scheduler),
      // so CTAs that finish early take the next unit of the longest-first list.
      // The next index is drawn when a unit starts and decoded (a binary
      // search over the scheduler's prefix sums) right after the unit's first
      // tile is requested, so neither latency sits between two units' loads.
      int* next_unit = p.ws + WsLayout{p.B, p.Hkv}.counters() + 1;
      int u = atomicAdd(next_unit, 1);
      Unit un{};
      if (u < h.n_units) un = decode_unit(p, h, u);
      while (ok && u < h.n_units) {
        const int u_next = atomicAdd(next_unit, 1);
        Unit nx = un;
        bool decoded = u_next >= h.n_units;
        un.u = u;
        un.last = 0;
        if (!(ok = publish(un))) break;
        const int nt = (un.ke - un.ks + TK - 1) / TK;
        for (int j = 0; j < nt; ++j, ++cnt) {
          const int st = cnt % C::STAGES;
          if (!(ok = mbar_wait(&empty[st], ((cnt / C::STAGES) & 1) ^ 1, abort, status))) break;
          const int k0 = tile_row<TK>(p, un, j, total_kv);
          uint8_t* dk = smem + C::OFF_KV + st * C::STAGE;
          mbar_arrive_expect_tx(&full[st], C::STAGE);
          load_kv_box(dk, &tmap_k, &full[st], p, 0, un.b, un.g, un.kv_start, k0);
          load_kv_box(dk + C::K_BYTES, &tmap_v, &full[st], p, 0, un.b, un.g, un.kv_start, k0);
          if (!decoded) {
            nx = decode_unit(p, h, u_next);
            decoded = true;
          }
        }
        if (!ok) break;
        if (!decoded) nx = decode_unit(p, h, u_next);
        u = u_next;
        un = nx;
      }
      if (ok) {
        Unit v{};
        v.last = 1;
        publish(v);
      }
      for (int s = 0; s < C::STAGES; ++s) {
        const uint32_t fills = cnt > (uint32_t)s ? (cnt - 1 - s) / C::STAGES + 1 : 0;
        if (fills) mbar_wait(&full[s], (fills - 1) & 1, abort, status);
      }
    }
  } else {
    // ------------------------------------------------------------ compute
    const int cw = warp - 1;  // compute warp 0 .. NW-1
    const int hgrp = cw / C::NWG, cwg = cw % C::NWG;  // head group, warp within it
    const int hbase = hgrp * GW;                       // first head of the group
    const float NEG_INF = __int_as_float(0xff800000);
    const bool capped = p.softcap != 0.0f;
    const float qmul = capped ? p.scale / p.softcap : p.scale * kLog2e;
    const float cap_mul = p.softcap * kLog2e;
    const int my_r = lane / GW;  // key of the (key, head) pair this lane owns after the reduce-scatter
    T* out = static_cast<T*>(p.out);
    uint32_t cnt = 0;
    bool ok = true;

    uint32_t taken = 0;
    while (ok) {
      const int usl = taken % kUnitSlots;
      ok = __all_sync(0xffffffffu, mbar_wait(&unit_full[usl], (taken / kUnitSlots) & 1, abort,
                                             status));
      if (!ok) break;
      const Unit un = units[usl];
      __syncwarp();
      if (lane == 0) mbar_arrive(&unit_empty[usl]);
      ++taken;
      if (un.last) break;
      const int u = un.u;
      const int nt = (un.ke - un.ks + TK - 1) / TK;

      float q[GW][DPLK];
      {
        const T* Q = static_cast<const T*>(p.q);
#pragma unroll
        for (int hh = 0; hh < GW; ++hh) {
          if (lane < C::LK) {
            const uint8_t* row = reinterpret_cast<const uint8_t*>(
                Q + ((size_t)un.q_tok * p.H + (size_t)un.g * G + hbase + hh) * DK);
            load_dims<T, DPLK>(row, lane, q[hh]);
          } else {
#pragma unroll
            for (int e = 0; e < DPLK; ++e) q[hh][e] = 0.0f;
          }
#pragma unroll
          for (int e = 0; e < DPLK; ++e) q[hh][e] *= qmul;
        }
      }
      float acc[GW][DPLV];
#pragma unroll
      for (int hh = 0; hh < GW; ++hh)
#pragma unroll
        for (int e = 0; e < DPLV; ++e) acc[hh][e] = 0.0f;
      float m_run = NEG_INF, l_part = 0.0f;

      for (int j = 0; j < nt; ++j, ++cnt) {
        const int st = cnt % C::STAGES;
        ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (cnt / C::STAGES) & 1, abort, status));
        if (!ok) break;
        const uint8_t* sK = smem + C::OFF_KV + st * C::STAGE;
        const uint8_t* sV = sK + C::K_BYTES;
        const int k0 = tile_row<TK>(p, un, j, total_kv);
        const int base = k0 - un.kv_start;            // local key of tile row 0
        const int lo = un.ks + j * TK - base;          // visible tile rows [lo, hi)
        const int hi = min(un.ks + (j + 1) * TK, un.ke) - base;
        // Rounds are dealt to the head group's warps across tiles: round rd
        // of tile j goes to warp (j * RPT + rd) mod NWG, so that with fewer
        // rounds per tile than warps (small G) the warps take whole tiles in
        // turn instead of leaving most of them idle.
        const int rd0 = ((cwg - j * C::RPT) % C::NWG + C::NWG) % C::NWG;
        for (int rd = rd0; rd < C::RPT; rd += C::NWG) {
          const int r0 = rd * R;  // first tile row of this round
          float v[32];
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float kf[DPLK];
            if (C::LK == 32 || lane < C::LK) {
              load_dims<T, DPLK>(sK + (size_t)(r0 + r) * DK * 2, lane, kf);
            } else {
#pragma unroll
              for (int e = 0; e < DPLK; ++e) kf[e] = 0.0f;
            }
#pragma unroll
            for (int hh = 0; hh < GW; ++hh) {
              float2 a = make_float2(0.0f, 0.0f);
#pragma unroll
              for (int e = 0; e < DPLK; e += 2)
                a = ffma2(make_float2(q[hh][e], q[hh][e + 1]), make_float2(kf[e], kf[e + 1]), a);
              v[r * GW + hh] = a.x + a.y;
            }
          }
          // reduce-scatter: after the 5 steps lane l holds the full dot of pair l
#pragma unroll
          for (int step = 16; step >= 1; step >>= 1) {
            const bool upper = (lane & step) != 0;
#pragma unroll
            for (int i = 0; i < step; ++i) {
              const float send = upper ? v[i] : v[i + step];
              const float keep = upper ? v[i + step] : v[i];
              v[i] = keep + __shfl_xor_sync(0xffffffffu, send, step);
            }
          }
          const int row = r0 + my_r;
          float x = capped ? cap_mul * tanh_via_exp2(v[0]) : v[0];
          x = (row >= lo && row < hi) ? x : NEG_INF;
          float mr = x;
#pragma unroll
          for (int o = GW; o < 32; o <<= 1) mr = fmaxf(mr, __shfl_xor_sync(0xffffffffu, mr, o));
          const float m_new = fmaxf(m_run, mr);
          float alpha = 1.0f, pr = 0.0f;
          if (m_new != NEG_INF) {
            alpha = ex2_approx(m_run - m_new);
            pr = ex2_approx(x - m_new);
          }
          m_run = m_new;
          l_part = l_part * alpha + pr;
          sP[cw * 32 + lane] = pr;
          if (lane < GW) sA[cw * GW + lane] = alpha;
          __syncwarp();
#pragma unroll
          for (int hh = 0; hh < GW; ++hh) {
            const float a = sA[cw * GW + hh];
#pragma unroll
            for (int e = 0; e < DPLV; ++e) acc[hh][e] *= a;
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            float vf[DPLV];
            if (C::LV == 32 || lane < C::LV) {
              load_dims<T, DPLV>(sV + (size_t)(r0 + r) * DV * 2, lane, vf);
            } else {
#pragma unroll
              for (int e = 0; e < DPLV; ++e) vf[e] = 0.0f;
            }
            float pw[GW];
            load_probs<GW>(sP + cw * 32 + r * GW, pw);
#pragma unroll
            for (int hh = 0; hh < GW; ++hh)
#pragma unroll
              for (int e = 0; e < DPLV; e += 2) {
                const float2 a = ffma2(make_float2(pw[hh], pw[hh]), make_float2(vf[e], vf[e + 1]),
                                       make_float2(acc[hh][e], acc[hh][e + 1]));
                acc[hh][e] = a.x;
                acc[hh][e + 1] = a.y;
              }
          }
          __syncwarp();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
      }

      // per-head sum over this warp's lanes, then merge the warps of each
      // head group
#pragma unroll
      for (int o = GW; o < 32; o <<= 1) l_part += __shfl_xor_sync(0xffffffffu, l_part, o);
      if (lane < GW) {
        sM[cw * GW + lane] = m_run;
        sL[cw * GW + lane] = l_part;
      }
      if (C::LV == 32 || lane < C::LV) {
#pragma unroll
        for (int hh = 0; hh < GW; ++hh)
#pragma unroll
          for (int e = 0; e < DPLV; ++e)
            sO[(cw * GW + hh) * DV + lane * DPLV + e] = acc[hh][e];
      }
      // Every compute warp reaches this barrier, whether it finished its tiles
      // or gave up on a wait; the give-up decision is then read by all of
      // them at once, so no warp is ever left alone at a named barrier.
      compute_bar_sync<C::NW>();
      if (*abort) break;

      const int t = threadIdx.x - 32;  // 0 .. 32 NW - 1
      const bool split = un.S > 1;
      float* part = p.partials + (size_t)u * (G * DV + 2 * G);
      for (int e = t; e < G * DV; e += C::NW * 32) {
        const int hh = e / DV;  // head within the kv group
        const int grp = hh / GW, lh = hh - grp * GW, de = e - hh * DV;
        const int w0 = grp * C::NWG;  // the warps that served this head
        float M = NEG_INF;
#pragma unroll
        for (int w = 0; w < C::NWG; ++w) M = fmaxf(M, sM[(w0 + w) * GW + lh]);
        float Lsum = 0.0f, O = 0.0f;
        if (M != NEG_INF) {
#pragma unroll
          for (int w = 0; w < C::NWG; ++w) {
            const float sc = ex2_approx(sM[(w0 + w) * GW + lh] - M);
            Lsum += sL[(w0 + w) * GW + lh] * sc;
            O += sO[((w0 + w) * GW + lh) * DV + de] * sc;
          }
        }
        if (!split) {
          const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
          out[((size_t)un.q_tok * p.H + (size_t)un.g * G) * DV + e] = static_cast<T>(O * inv);
        } else {
          part[e] = O;
          if (de == 0) {
            part[G * DV + hh] = M;
            part[G * DV + G + hh] = Lsum;
          }
        }
      }
      if (split) {
        __threadfence();
        compute_bar_sync<C::NW>();
        if (t == 0) {
          const WsLayout L{p.B, p.Hkv};
          int* done = p.ws + L.dec_done() + (size_t)un.b * p.Hkv + un.g;
          s_last = atomicAdd(done, 1) == un.S - 1;
        }
        compute_bar_sync<C::NW>();
        if (s_last) {
          __threadfence();
          const float* first = p.partials + (size_t)(u - un.s) * (G * DV + 2 * G);
          const size_t stride = G * DV + 2 * G;
          for (int e = t; e < G * DV; e += C::NW * 32) {
            const int hh = e / DV;
            float M = NEG_INF;
            for (int s = 0; s < un.S; ++s) M = fmaxf(M, __ldcg(first + s * stride + G * DV + hh));
            float Lsum = 0.0f, O = 0.0f;
            if (M != NEG_INF) {
              for (int s = 0; s < un.S; ++s) {
                const float* ps = first + s * stride;
                const float sc = ex2_approx(__ldcg(ps + G * DV + hh) - M);
                Lsum += __ldcg(ps + G * DV + G + hh) * sc;
                O += __ldcg(ps + e) * sc;
              }
            }
            const float inv = Lsum > 0.0f ? 1.0f / Lsum : 0.0f;
            out[((size_t)un.q_tok * p.H + (size_t)un.g * G) * DV + e] = static_cast<T>(O * inv);
          }
        }
      }
      compute_bar_sync<C::NW>();  // shared merge buffers are reused by the next unit
    }
  }
  __syncthreads();
}

template <typename T, int DK, int DV, int G>
cudaError_t launch_dec(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                       int num_sms, cudaStream_t s) {
  constexpr int smem = DecCfg<DK, DV, G>::SMEM;
  auto kern = pva_decode_kernel<T, DK, DV, G>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  return launch_dependent(kern, dim3(num_sms), dim3(DecCfg<DK, DV, G>::THREADS), smem, s, p, tk,
                          tv);
}

template <typename T, int DK, int DV>
cudaError_t launch_dec_g(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                         int num_sms, cudaStream_t s) {
  switch (p.G) {
    case 1: return launch_dec<T, DK, DV, 1>(p, tk, tv, num_sms, s);
    case 2: return launch_dec<T, DK, DV, 2>(p, tk, tv, num_sms, s);
    case 4: return launch_dec<T, DK, DV, 4>(p, tk, tv, num_sms, s);
    case 8: return launch_dec<T, DK, DV, 8>(p, tk, tv, num_sms, s);
    case 16: return launch_dec<T, DK, DV, 16>(p, tk, tv, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t launch_dec_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv,
                         int num_sms, cudaStream_t s) {
  if (p.d == p.dv) {
    switch (p.d) {
      case 64: return launch_dec_g<T, 64, 64>(p, tk, tv, num_sms, s);
      case 96: return launch_dec_g<T, 96, 96>(p, tk, tv, num_sms, s);
      case 128: return launch_dec_g<T, 128, 128>(p, tk, tv, num_sms, s);
      case 192: return launch_dec_g<T, 192, 192>(p, tk, tv, num_sms, s);
      case 256: return launch_dec_g<T, 256, 256>(p, tk, tv, num_sms, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.d == 192 && p.dv == 128) return launch_dec_g<T, 192, 128>(p, tk, tv, num_sms, s);
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_decode(const AttnParams& p, int dtype, const CUtensorMap& tk,
                          const CUtensorMap& tv, int num_sms, cudaStream_t s) {
  return dtype == PVA_BF16 ? launch_dec_t<__nv_bfloat16>(p, tk, tv, num_sms, s)
                           : launch_dec_t<__half>(p, tk, tv, num_sms, s);
}

}  // namespace pva
