// On-device tile scheduler.
//
// Turns cu_seqlens_q / cu_seqlens_kv (packed_varlen_attention.rs, "Packed
// layout & cumulative offsets") into the work description the compute
// kernels read, without copying anything back to the host:
//
//   * validation of the offsets (start at 0, non-decreasing -- the checks the
//     page's `execute` performs on the host), latched as status bits; on any
//     error the work lists are left empty so nothing is written;
//   * a prefill list: sequences with L_q > 0 (L_q >= 2 when decode routing is
//     on), longest key range first (ties by sequence index), with an inclusive
//     prefix of their work-item counts ceil(L_q / tile_tokens) * units;
//   * a decode list: sequences with L_q == 1 (when routing is on), longest
//     first, each split into S_b key chunks, with a prefix of their
//     (kv head, split) unit counts;
//   * zeroed split-completion counters for the decode combine, and zeroed
//     work counters from which the persistent compute kernels draw items.
//
// One warp for B <= 32 (everything in registers), else one CTA of 128, 512 or
// 1024 threads (by B).  Up to 16384 sequences are sorted in (dynamic) shared
// memory (a rank sort up to 512, bitonic above); larger batches keep their
// input order.
#include <limits.h>

#include "pva_device.cuh"

namespace pva {

namespace {


// Exclusive scan of one int64 per thread across the CTA of NT threads;
// returns the exclusive prefix and writes the CTA total to *total.
template <int NT>
__device__ long long block_exclusive_scan(long long v, long long* scratch, long long* total) {
  constexpr int NW = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    long long y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    long long w = lane < NW ? scratch[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      long long y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    scratch[lane] = w;  // inclusive per-warp totals
  }
  __syncthreads();
  const long long warp_base = warp ? scratch[warp - 1] : 0;
  const long long tot = scratch[NW - 1];
  __syncthreads();
  *total = tot;
  return warp_base + x - v;
}

template <int NT>
__device__ long long block_sum(long long v, long long* scratch) {
  long long t;
  block_exclusive_scan<NT>(v, scratch, &t);
  return t;
}

struct SeqLens {
  int lq, lkv;
};

// Per-sequence lengths: from shared memory when the batch was staged there
// (B <= kStageMax: one coalesced pass over the offsets), else from global.
struct Lengths {
  const int32_t* cu_q;
  const int32_t* cu_kv;
  const int32_t* kv_len;  // padded K/V lengths, or nullptr
  const int* s_lq;   // nullptr when not staged
  const int* s_lkv;
  __device__ __forceinline__ SeqLens operator()(int b) const {
    if (s_lq) return SeqLens{s_lq[b], s_lkv[b]};
    return SeqLens{cu_q[b + 1] - cu_q[b], kv_len ? kv_len[b] : cu_kv[b + 1] - cu_kv[b]};
  }
};

// Keys a single-row (decode) sequence attends to: all L_kv, or the last W of
// them under a local window W.
__device__ __forceinline__ int decode_keys(int lkv, int window) {
  return window > 0 && window < lkv ? window : lkv;
}

__device__ __forceinline__ int decode_splits(int lkv, int chunk) {
  if (lkv <= chunk) return 1;
  int s = (lkv + chunk - 1) / chunk;
  return s < kDecodeMaxSplits ? s : kDecodeMaxSplits;
}

// Builds one ordered list (class 0 = prefill, 1 = decode) and its prefix.
// Returns false when the work count overflows int32.
// When the batch is sorted (B <= kSortMax) the sorted list is also kept in
// shared memory (s_order), so the prefix pass never reads back global memory.
template <int NT>
__device__ bool build_list(const AttnParams& p, const SchedConfig& c, const Lengths& seq_lens,
                           int cls, int chunk, bool dec_route, int32_t* order, int32_t* prefix,
                           int* n_out, int* total_out, unsigned long long* keys, int32_t* s_order,
                           long long* scratch) {
  const int B = p.B;
  auto member = [&](int b) -> bool {
    SeqLens s = seq_lens(b);
    if (s.lq <= 0) return false;
    const bool is_dec = dec_route && s.lq == 1;
    return cls == 1 ? is_dec : !is_dec;
  };
  auto work = [&](int b) -> long long {
    SeqLens s = seq_lens(b);
    if (cls == 0)
      return (long long)((s.lq + c.tile_tokens - 1) / c.tile_tokens) * c.units_per_tile;
    return (long long)decode_splits(decode_keys(s.lkv, p.window), chunk) * p.Hkv;
  };

  int n = 0;
  if (B <= kSortMax) {
    // An empty list (a batch of only prefill or only decode rows) skips the
    // sort; its order and prefix are written as the sort would leave them.
    long long members = 0;
    for (int b = threadIdx.x; b < B; b += NT) members += member(b);
    members = block_sum<NT>(members, scratch);
    if (members == 0) {
      for (int i = threadIdx.x; i < B; i += NT) order[i] = -1;
      for (int i = threadIdx.x; i <= B; i += NT) prefix[i] = 0;
      *n_out = 0;
      *total_out = 0;
      return true;
    }
    auto sort_key = [&](int i) -> unsigned long long {
      if (!member(i)) return ~0ull;
      SeqLens s = seq_lens(i);
      return ((unsigned long long)(unsigned)(INT_MAX - s.lkv) << 32) | (unsigned)i;
    };
    if (B <= 512 && B <= NT) {
      // Rank sort, one thread per sequence: a member's place is the number
      // of members with a smaller key (keys are unique: the sequence index
      // breaks ties; non-members hold the largest key), found in one pass
      // over the keys in shared memory between two barriers instead of the
      // bitonic network's log2(N) (log2(N) + 1) / 2 barriered steps (B = 256
      // took about 22000 cycles for this list that way).
      for (int i = threadIdx.x; i < B; i += NT) keys[i] = sort_key(i);
      __syncthreads();
      const int i = threadIdx.x;
      if (i < B) {
        const unsigned long long me = keys[i];
        if (me != ~0ull) {
          int rank = 0;
#pragma unroll 4
          for (int j = 0; j < B; ++j) rank += keys[j] < me ? 1 : 0;
          order[rank] = i;
          s_order[rank] = i;
        }
      }
      n = (int)members;
      for (int j = n + threadIdx.x; j < B; j += NT) {
        order[j] = -1;
        s_order[j] = -1;
      }
    } else {
      int N = 1;
      while (N < B) N <<= 1;
      for (int i = threadIdx.x; i < N; i += NT) keys[i] = i < B ? sort_key(i) : ~0ull;
      __syncthreads();
      for (int k = 2; k <= N; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
          for (int i = threadIdx.x; i < N; i += NT) {
            const int ixj = i ^ j;
            if (ixj > i) {
              const unsigned long long a = keys[i], bb = keys[ixj];
              const bool up = (i & k) == 0;
              if ((a > bb) == up) {
                keys[i] = bb;
                keys[ixj] = a;
              }
            }
          }
          __syncthreads();
        }
      }
      for (int i = threadIdx.x; i < B; i += NT) {
        const bool valid = keys[i] != ~0ull;
        const int32_t o = valid ? (int32_t)(keys[i] & 0xffffffffu) : -1;
        order[i] = o;
        s_order[i] = o;
      }
      n = (int)members;
    }
  } else {
    // Input order: compact the members with a scan over contiguous chunks.
    const int per = (B + NT - 1) / NT;
    const int lo = min(B, (int)threadIdx.x * per), hi = min(B, lo + per);
    long long local = 0;
    for (int b = lo; b < hi; ++b) local += member(b);
    long long total;
    long long pos = block_exclusive_scan<NT>(local, scratch, &total);
    for (int b = lo; b < hi; ++b)
      if (member(b)) order[pos++] = b;
    __syncthreads();
    n = (int)total;
    for (int i = n + threadIdx.x; i < B; i += NT) order[i] = -1;
  }
  __syncthreads();

  // Prefix of work counts in list order: contiguous chunk per thread.
  const int32_t* lst = B <= kSortMax ? s_order : order;
  const int per = (n + NT - 1) / NT;
  const int lo = min(n, (int)threadIdx.x * per), hi = min(n, lo + per);
  long long local = 0;
  for (int i = lo; i < hi; ++i) local += work(lst[i]);
  long long total;
  long long run = block_exclusive_scan<NT>(local, scratch, &total);
  const bool fits = total <= (long long)INT_MAX;
  if (fits) {
    for (int i = lo; i < hi; ++i) {
      prefix[i] = (int32_t)run;
      run += work(lst[i]);
    }
    for (int i = n + threadIdx.x; i <= B; i += NT) prefix[i] = (int32_t)total;
  }
  *n_out = n;
  *total_out = fits ? (int)total : 0;
  return fits;
}

// NT threads: the smallest of 128, 512, 1024 that covers B (a small batch
// does not pay for 32 warps walking through every barrier and scan).
// Dynamic shared memory of the CTA scheduler for a batch of B sequences:
// sort keys [next power of two >= B] (u64), the sorted list [B], and, for
// B <= kStageMax, the staged lengths [B] x 2.  Zero when B > kSortMax.
__host__ __device__ inline size_t sched_smem_bytes(int B) {
  if (B > kSortMax) return 0;
  size_t N = 1;
  while (N < (size_t)B) N <<= 1;
  return N * 8 + (size_t)B * 4 * (B <= kStageMax ? 3 : 1);
}

template <int NT>
__global__ void __launch_bounds__(NT) pva_schedule_kernel(AttnParams p, SchedConfig c) {
  extern __shared__ unsigned long long dyn_smem[];
  size_t N = 1;
  while (N < (size_t)p.B) N <<= 1;
  unsigned long long* keys = dyn_smem;
  int32_t* s_order = reinterpret_cast<int32_t*>(keys + N);
  int* s_lq = s_order + p.B;
  int* s_lkv = s_lq + p.B;
  __shared__ long long scratch[32];
  __shared__ uint32_t s_status;
  __shared__ int s_chunk;

  // The compute kernels are launched as programmatic dependents: let them
  // start their set-up now; they wait for this grid before reading its output.
  // This grid is one too (its launch overlaps the end of the work before it),
  // so it waits for that work before reading the offsets.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  wait_prior_grid();

  const int B = p.B;
  const WsLayout L{B, p.Hkv};
  int32_t* ws = p.ws;
  SchedHeader* hdr = reinterpret_cast<SchedHeader*>(ws + kWsHeader);
  const bool staged = B <= kStageMax;
  const Lengths seq_lens{p.cu_q, p.cu_kv, p.kv_len, staged ? s_lq : nullptr,
                         staged ? s_lkv : nullptr};

  if (threadIdx.x == 0) s_status = 0;
  __syncthreads();
  // One pass over the offsets (all loads in flight together).
  if (threadIdx.x == 0) {
    uint32_t st = 0;
    if (p.cu_q[0] != 0) st |= PVA_DEV_CU_Q_START;
    if (p.cu_kv[0] != 0) st |= PVA_DEV_CU_KV_START;
    // Empty tensors may come as NULL; a NULL with a nonzero extent may not.
    if ((!p.q || !p.out) && p.cu_q[B] != 0) st |= PVA_DEV_NULL_TENSOR;
    if ((!p.k || !p.v) && p.cu_kv[B] != 0) st |= PVA_DEV_NULL_TENSOR;
    if (st) atomicOr(&s_status, st);
  }
  for (int b = threadIdx.x; b < B; b += NT) {
    const int lq = p.cu_q[b + 1] - p.cu_q[b];
    const int slot = p.cu_kv[b + 1] - p.cu_kv[b];
    const int lkv = p.kv_len ? p.kv_len[b] : slot;
    if (lq < 0) atomicOr(&s_status, PVA_DEV_CU_Q_ORDER);
    if (slot < 0) atomicOr(&s_status, PVA_DEV_CU_KV_ORDER);
    // (a cache step the front end rejected comes with -1 lengths and has
    // latched its own bit already)
    if (lkv < 0 || lkv > slot) atomicOr(&s_status, p.kv_cap ? PVA_DEV_KV_CACHE : PVA_DEV_KV_LEN);
    if (staged) {
      s_lq[b] = lq;
      s_lkv[b] = lkv;
    }
  }
  // Completion counters of the decode combine start at zero every call.
  int32_t* done = ws + L.dec_done();
  for (long long i = threadIdx.x; i < (long long)B * p.Hkv; i += NT) done[i] = 0;
  if (threadIdx.x < 4) ws[L.counters() + threadIdx.x] = 0;  // work counters of this call
  __syncthreads();

  int n_pref = 0, n_items = 0, n_dec = 0, n_units = 0;
  if (s_status == 0) {
    // Whether single-row sequences go to the split-KV decode kernel (see
    // SchedConfig::decode_adaptive).
    bool dec_route = c.decode_enabled != 0;
    if (dec_route && c.decode_adaptive) {
      long long single = 0;
      for (int b = threadIdx.x; b < B; b += NT) single += seq_lens(b).lq == 1;
      single = block_sum<NT>(single, scratch);
      dec_route = single * p.Hkv < 2LL * c.num_sms;
    }
    // Decode chunk: aim for about 2 units per SM (every split costs a unit's
    // start, its merge, an fp32 partial and the combine: 8 per SM measured
    // 6-16% slower on 8 to 128 sequences, and the same at 256, where neither
    // splits), never more partial slots than the workspace holds (all
    // sequences unsplit if it must).
    if (dec_route) {
      long long keyrows = 0, cnt = 0;
      for (int b = threadIdx.x; b < B; b += NT) {
        SeqLens s = seq_lens(b);
        if (s.lq == 1) {
          keyrows += decode_keys(s.lkv, p.window);
          cnt += 1;
        }
      }
      keyrows = block_sum<NT>(keyrows, scratch) * p.Hkv;
      cnt = block_sum<NT>(cnt, scratch);
      long long target = (long long)c.num_sms * 2;
      long long chunk = (keyrows + target - 1) / target;
      chunk = ((chunk + 63) / 64) * 64;
      if (chunk < 256) chunk = 256;
      // grow the chunk until the split units fit the partial slots
      for (int it = 0; it < 40; ++it) {
        long long units = 0;
        for (int b = threadIdx.x; b < B; b += NT) {
          SeqLens s = seq_lens(b);
          if (s.lq == 1) {
            int sp = decode_splits(decode_keys(s.lkv, p.window),
                                   chunk > INT_MAX ? INT_MAX : (int)chunk);
            units += (long long)sp * p.Hkv;
          }
        }
        units = block_sum<NT>(units, scratch);
        // one unit per (sequence, kv head) means that nothing is split
        if (units == cnt * p.Hkv || units <= p.dec_cap_units) break;
        chunk *= 2;
      }
      if (threadIdx.x == 0) s_chunk = chunk > INT_MAX ? INT_MAX : (int)chunk;
    } else if (threadIdx.x == 0) {
      s_chunk = INT_MAX;
    }
    __syncthreads();
    const int chunk = s_chunk;
    bool ok = build_list<NT>(p, c, seq_lens, 0, chunk, dec_route, ws + L.pref_order(),
                             ws + L.pref_prefix(), &n_pref, &n_items, keys, s_order, scratch);
    __syncthreads();
    ok = build_list<NT>(p, c, seq_lens, 1, chunk, dec_route, ws + L.dec_order(),
                        ws + L.dec_prefix(), &n_dec, &n_units, keys, s_order, scratch) && ok;
    if (!ok) {
      if (threadIdx.x == 0) atomicOr(&s_status, PVA_DEV_TOO_MANY);
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const uint32_t st = s_status;
    SchedHeader h;
    h.status = st;
    h.n_pref = st ? 0 : n_pref;
    h.n_items = st ? 0 : n_items;
    h.n_dec = st ? 0 : n_dec;
    h.n_units = st ? 0 : n_units;
    h.tile_tokens = c.tile_tokens;
    h.units_per_tile = c.units_per_tile;
    h.dec_chunk = st ? 0 : s_chunk;
    *hdr = h;
    if (st) atomicOr(p.status, st);
  }
}

// Warp-level sums (long long) over the 32 lanes.
__device__ __forceinline__ long long warp_sum_ll(long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// The same scheduler for B <= 32, in one warp: sequence b lives in lane b,
// the two lists are sorted with a bitonic network over the lanes (shuffles)
// and their prefixes are warp scans.  Nothing goes through shared memory or
// CTA barriers, which dominate the CTA version at small B; the work lists,
// counters and status bits are identical.
__global__ void __launch_bounds__(32) pva_schedule_warp_kernel(AttnParams p, SchedConfig c) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  wait_prior_grid();  // launched as a dependent of the work before it
  const unsigned full = 0xffffffffu;
  const int lane = threadIdx.x, B = p.B;
  const WsLayout L{B, p.Hkv};
  int32_t* ws = p.ws;
  const bool mine = lane < B;

  uint32_t st = 0;
  int lq = 0, lkv = 0;
  if (mine) {
    lq = p.cu_q[lane + 1] - p.cu_q[lane];
    const int slot = p.cu_kv[lane + 1] - p.cu_kv[lane];
    lkv = p.kv_len ? p.kv_len[lane] : slot;
    if (lq < 0) st |= PVA_DEV_CU_Q_ORDER;
    if (slot < 0) st |= PVA_DEV_CU_KV_ORDER;
    if (lkv < 0 || lkv > slot) st |= p.kv_cap ? PVA_DEV_KV_CACHE : PVA_DEV_KV_LEN;
  }
  if (lane == 0) {
    if (p.cu_q[0] != 0) st |= PVA_DEV_CU_Q_START;
    if (p.cu_kv[0] != 0) st |= PVA_DEV_CU_KV_START;
    if ((!p.q || !p.out) && p.cu_q[B] != 0) st |= PVA_DEV_NULL_TENSOR;
    if ((!p.k || !p.v) && p.cu_kv[B] != 0) st |= PVA_DEV_NULL_TENSOR;
  }
  st = __reduce_or_sync(full, st);
  int32_t* done = ws + L.dec_done();
  for (int i = lane; i < B * p.Hkv; i += 32) done[i] = 0;
  if (lane < 4) ws[L.counters() + lane] = 0;

  int n_pref = 0, n_items = 0, n_dec = 0, n_units = 0, chunk = INT_MAX;
  if (st == 0) {
    bool dec_route = c.decode_enabled != 0;
    if (dec_route && c.decode_adaptive)
      dec_route = (long long)__popc(__ballot_sync(full, mine && lq == 1)) * p.Hkv <
                  2LL * c.num_sms;
    const bool is_dec = mine && dec_route && lq == 1;
    if (dec_route) {
      const long long keyrows = warp_sum_ll(is_dec ? decode_keys(lkv, p.window) : 0) * p.Hkv;
      const long long target = (long long)c.num_sms * 2;
      long long ch = (keyrows + target - 1) / target;
      ch = ((ch + 63) / 64) * 64;
      if (ch < 256) ch = 256;
      for (int it = 0; it < 40; ++it) {
        const int sp =
            is_dec ? decode_splits(decode_keys(lkv, p.window), ch > INT_MAX ? INT_MAX : (int)ch)
                   : 0;
        const long long units = warp_sum_ll((long long)sp * p.Hkv);
        if (!__any_sync(full, sp > 1) || units <= p.dec_cap_units) break;
        ch *= 2;
      }
      chunk = ch > INT_MAX ? INT_MAX : (int)ch;
    }
    bool ok = true;
#pragma unroll 1
    for (int cls = 0; cls < 2; ++cls) {
      const bool member = mine && lq > 0 && (cls == 1 ? is_dec : !is_dec);
      unsigned long long key =
          member ? ((unsigned long long)(unsigned)(INT_MAX - lkv) << 32) | (unsigned)lane : ~0ull;
#pragma unroll
      for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
        for (int j = k >> 1; j > 0; j >>= 1) {
          const unsigned long long other = __shfl_xor_sync(full, key, j);
          const unsigned long long lo = key < other ? key : other, hi = key < other ? other : key;
          key = (((lane & j) == 0) == ((lane & k) == 0)) ? lo : hi;
        }
      const int n = __popc(__ballot_sync(full, member));
      const int o = key != ~0ull ? (int)(key & 0xffffffffu) : -1;
      int32_t* order = ws + (cls == 0 ? L.pref_order() : L.dec_order());
      int32_t* prefix = ws + (cls == 0 ? L.pref_prefix() : L.dec_prefix());
      if (mine) order[lane] = o;
      const int lq_o = __shfl_sync(full, lq, o & 31), lkv_o = __shfl_sync(full, lkv, o & 31);
      long long w = 0;
      if (lane < n)
        w = cls == 0 ? (long long)((lq_o + c.tile_tokens - 1) / c.tile_tokens) * c.units_per_tile
                     : (long long)decode_splits(decode_keys(lkv_o, p.window), chunk) * p.Hkv;
      long long incl = w;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const long long y = __shfl_up_sync(full, incl, d);
        if (lane >= d) incl += y;
      }
      const long long total = __shfl_sync(full, incl, 31);
      const bool fits = total <= (long long)INT_MAX;
      if (fits) {
        if (lane < n) prefix[lane] = (int32_t)(incl - w);
        for (int i = n + lane; i <= B; i += 32) prefix[i] = (int32_t)total;
      }
      ok = ok && fits;
      if (cls == 0) {
        n_pref = n;
        n_items = fits ? (int)total : 0;
      } else {
        n_dec = n;
        n_units = fits ? (int)total : 0;
      }
    }
    if (!ok) st |= PVA_DEV_TOO_MANY;
  }
  if (lane == 0) {
    SchedHeader h;
    h.status = st;
    h.n_pref = st ? 0 : n_pref;
    h.n_items = st ? 0 : n_items;
    h.n_dec = st ? 0 : n_dec;
    h.n_units = st ? 0 : n_units;
    h.tile_tokens = c.tile_tokens;
    h.units_per_tile = c.units_per_tile;
    h.dec_chunk = st ? 0 : chunk;
    *reinterpret_cast<SchedHeader*>(ws + kWsHeader) = h;
    if (st) atomicOr(p.status, st);
  }
}

}  // namespace

// Front end of pva_forward_padded: the padded layout as packed offsets.  Batch
// b's queries are rows [b q_seq, (b+1) q_seq) and its key/value slot rows
// [b kv_seq, (b+1) kv_seq), of which the first nonpad[b] are its keys (the
// exclusive prefix sum of the pages' nonpad_kv_seqlen, taken over slots
// instead of over packed keys, so nothing is copied).  A length outside
// [0, kv_seq] is stored as -1, which the scheduler reports as PVA_DEV_KV_LEN.
__global__ void pva_padded_front_kernel(const int64_t* nonpad, int B, int q_seq, int kv_seq,
                                        int32_t* cu_q, int32_t* cu_kv, int32_t* kv_len) {
  // a programmatic dependent of the work before it, like every kernel here
  allow_next_grid();
  wait_prior_grid();
  for (int b = blockIdx.x * blockDim.x + threadIdx.x; b <= B; b += gridDim.x * blockDim.x) {
    cu_q[b] = b * q_seq;
    cu_kv[b] = b * kv_seq;
    if (b < B) {
      const long long n = nonpad[b];
      kv_len[b] = (n < 0 || n > kv_seq) ? -1 : (int32_t)n;
    }
  }
}

cudaError_t launch_padded_front(const int64_t* nonpad, int B, int q_seq, int kv_seq,
                                int32_t* cu_q, int32_t* cu_kv, int32_t* kv_len, cudaStream_t s) {
  const int threads = 256, blocks = (B + threads) / threads;
  return launch_dependent(pva_padded_front_kernel, dim3(blocks < 1024 ? blocks : 1024),
                          dim3(threads), 0, s, nonpad, B, q_seq, kv_seq, cu_q, cu_kv, kv_len);
}

cudaError_t launch_scheduler(const AttnParams& p, const SchedConfig& c, cudaStream_t s) {
  // Programmatic dependents of the work before them (each waits for it first).
  if (p.B <= 32)
    return launch_dependent(pva_schedule_warp_kernel, dim3(1), dim3(32), 0, s, p, c);
  if (p.B <= 128)
    return launch_dependent(pva_schedule_kernel<128>, dim3(1), dim3(128), sched_smem_bytes(p.B),
                            s, p, c);
  if (p.B <= 512)
    return launch_dependent(pva_schedule_kernel<512>, dim3(1), dim3(512), sched_smem_bytes(p.B),
                            s, p, c);
  // more than 48 KB of dynamic shared memory needs the opt-in
  cudaError_t e = cudaFuncSetAttribute(pva_schedule_kernel<1024>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)sched_smem_bytes(kSortMax));
  if (e != cudaSuccess) return e;
  return launch_dependent(pva_schedule_kernel<1024>, dim3(1), dim3(1024),
                          sched_smem_bytes(p.B), s, p, c);
}

}  // namespace pva

// ---------------------------------------------------------------------------
// Self-test of the bounded waits: one CTA waits on an mbarrier that nothing
// ever completes, through the same helper every pipeline wait uses, with a
// short limit.  The wait gives up, latches PVA_DEV_WAIT_TIMEOUT and the kernel
// returns normally, leaving the context usable.
// ---------------------------------------------------------------------------
namespace pva {
namespace {

__global__ void pva_wait_selftest_kernel(uint32_t* status, uint64_t limit_ns, int* done) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    abort_flag = 0;
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  // Nobody arrives on `bar`: every thread's wait must run out.
  const bool ok = mbar_wait(&bar, 0, &abort_flag, status, limit_ns);
  __syncthreads();
  if (threadIdx.x == 0) *done = ok ? 1 : 2;
}

}  // namespace

cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, int* done, cudaStream_t s) {
  pva_wait_selftest_kernel<<<1, 64, 0, s>>>(status, limit_ns, done);
  return cudaGetLastError();
}

}  // namespace pva
