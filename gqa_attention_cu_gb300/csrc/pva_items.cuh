// Decoding of a work-item index into (sequence, query tile, unit) using the
// scheduler's ordered list and prefix sums.  Every role of every kernel
// decodes the same index the same way, so no item descriptor is stored.
#pragma once

#include "pva_internal.h"

namespace pva {

struct PrefillItem {
  int b;         // sequence
  int t;         // query tile within the sequence (tiles run last to first)
  int unit;      // kv head (tensor-core kernel) or query head (fp32 kernel)
  int q_start;   // cu_seqlens_q[b]
  int kv_start;  // cu_seqlens_kv[b]
  int lq, lkv;   // sequence lengths
};

// Largest p in [0, n) with prefix[p] <= it (prefix strictly increasing).
__device__ __forceinline__ int find_segment(const int32_t* prefix, int n, int it) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= it) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Item `it` of the longest-first list: the sequences in pref_order, each
// contributing (query tiles x units) items.  Within a sequence the default
// order is query tile major (latest, most expensive tile first, all units of
// it); unit_major walks one unit's tiles after another instead, which keeps
// the K/V of few units hot in L2 when every unit has its own K/V (G = 1).
__device__ __forceinline__ PrefillItem decode_prefill_item(const AttnParams& p,
                                                           const SchedHeader& h, int it,
                                                           bool unit_major = false) {
  const WsLayout L{p.B, p.Hkv};
  const int32_t* order = p.ws + L.pref_order();
  const int32_t* prefix = p.ws + L.pref_prefix();
  const int pos = find_segment(prefix, h.n_pref, it);
  const int local = it - prefix[pos];
  PrefillItem r;
  r.b = order[pos];
  r.q_start = p.cu_q[r.b];
  r.kv_start = p.cu_kv[r.b];
  // (padded K/V: the sequence's keys are the first kv_len[b] of its slot)
  r.lq = p.cu_q[r.b + 1] - r.q_start;
  r.lkv = p.kv_len ? p.kv_len[r.b] : p.cu_kv[r.b + 1] - r.kv_start;
  const int n_tiles = (r.lq + h.tile_tokens - 1) / h.tile_tokens;
  if (unit_major) {
    // one unit's query tiles after another (latest first within each), so
    // that the CTAs running at the same time read the same unit's K/V
    r.unit = local / n_tiles;
    r.t = n_tiles - 1 - (local - r.unit * n_tiles);
  } else {
    const int rank = local / h.units_per_tile;
    r.unit = local - rank * h.units_per_tile;
    r.t = n_tiles - 1 - rank;  // most expensive (latest) query tile first
  }
  return r;
}

// K/V addressing.  Packed K/V [tokens, Hkv, d]: key row k0 (a token index)
// of kv head g sits at TMA coordinates (y, z) = (g, k0).  BNSH cache: plane
// b * Hkv + g, row k0 - kv_start, so (y, z) = (k0 - kv_start, b * Hkv + g).
__device__ __forceinline__ int2 kv_tma_yz(const AttnParams& p, int b, int g, int kv_start,
                                          int k0) {
  return p.kv_cap ? make_int2(k0 - kv_start, b * p.Hkv + g) : make_int2(g, k0);
}

// Largest token index + 1 a key tile may reach.  Packed tiles are clamped
// inside the tensor; a cache plane or padded slot is zero-filled past its end
// by the tensor copy, so those tiles are never shifted for the tensor's sake
// (the host keeps (B + 1) * kv_cap and B * kv_slot within int32).
__device__ __forceinline__ int kv_tile_end(const AttnParams& p) {
  return p.kv_cap || p.kv_slot ? INT_MAX : p.cu_kv[p.B];
}

// End (exclusive packed row) a sequence's key tiles are shifted back to.
// Packed K/V: the end of the tensor.  Cache planes and padded slots: the
// sequence's last key, so that its last tile ends there (starting before row
// 0 of its plane or slot, where the tensor copy reads zeros, for a sequence
// shorter than a tile) and no row past its keys -- whatever the cache or the
// padding holds there, NaN included -- is ever loaded.  Columns a shifted
// tile repeats are masked as already seen.
__device__ __forceinline__ int key_tile_limit(const AttnParams& p, int kv_start, int lkv,
                                              int total_kv) {
  return p.kv_cap || p.kv_slot ? kv_start + lkv : total_kv;
}

// Loads the box of `map` at column x holding key rows [k0, ...) (packed row
// index) of kv head g of sequence b, whose keys start at packed row
// kv_start: rank-3 (packed K/V or cache planes) or rank-4 (padded slots).
__device__ __forceinline__ void load_kv_box(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            const AttnParams& p, int x, int b, int g,
                                            int kv_start, int k0) {
  if (p.kv_slot) {
    tma_load_4d(dst, map, bar, x, g, k0 - kv_start, b);
  } else {
    const int2 yz = kv_tma_yz(p, b, g, kv_start, k0);
    tma_load_3d(dst, map, bar, x, yz.x, yz.y);
  }
}

// Row index (in units of head rows) of local key j of kv head g, sequence b.
__device__ __forceinline__ size_t kv_row(const AttnParams& p, int b, int kv_start, int g, int j) {
  return p.kv_cap ? (size_t)(b * p.Hkv + g) * p.kv_cap + j : (size_t)(kv_start + j) * p.Hkv + g;
}

// First local key an item must visit: 0, or with a local window W the window
// start of its first query row (later rows start later).
__device__ __forceinline__ int item_key_begin(const PrefillItem& it, int tile_tokens, int window) {
  if (window <= 0) return 0;
  const int first_row = it.t * tile_tokens;
  const int lo = first_row + (it.lkv - it.lq) + 1 - window;
  return lo > 0 ? lo : 0;
}

// End of the local key range an item must visit: keys beyond the causal
// frontier of its last query row are never loaded.
__device__ __forceinline__ int item_key_extent(const PrefillItem& it, int tile_tokens,
                                               int is_causal) {
  const int last_row = min((it.t + 1) * tile_tokens, it.lq) - 1;
  int hi = it.lkv;
  if (is_causal) hi = min(it.lkv, last_row + (it.lkv - it.lq) + 1);
  return hi > 0 ? hi : 0;
}

}  // namespace pva
