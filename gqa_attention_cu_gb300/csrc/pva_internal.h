// Internal definitions shared by the host launcher and the kernels of libpva:
// the workspace layout written by the on-device scheduler, the parameter
// block every kernel receives, tile constants and the launch functions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>
#include <type_traits>

#include "pva.h"

#define PVA_WAIT_LIMIT_NS 2000000000ull  // 2 s: no legitimate pipeline wait comes close
#define PVA_WAIT_SLICE_NS 100000u        // longest single sleep of a waiting thread (0.1 ms)

namespace pva {

// ---- tile shapes ------------------------------------------------------------
constexpr int kTcRows = 128;        // MMA rows per query tile (G heads x tokens)
constexpr int kF32TileTokens = 16;  // query tokens per fp32 work item
constexpr int kF32KeyTile = 32;     // keys per fp32 key/value tile
constexpr int kDecodeMaxSplits = 16;
constexpr int kDecodeMaxGroup = 16;  // largest H/Hkv served by the split-KV decode kernel
constexpr int kSortMax = 16384;     // sequences sorted on device; more keep input order
constexpr int kStageMax = 4096;     // sequence lengths staged in shared memory by the scheduler

// Query tiles per prefill work item: two 128-row tiles share each K/V tile
// in the paired kernel; one tile otherwise (TMEM holds one wide O).
// The paired kernel (two query tiles per item) takes d == dv in {64, 128};
// every other tensor-core shape runs one tile per item.
__host__ __device__ constexpr bool tc_paired(int d, int dv) { return d == dv && (d == 64 || d == 128); }
__host__ __device__ constexpr int tc_tiles_per_item(int d, int dv) { return tc_paired(d, dv) ? 2 : 1; }
// Keys per tensor-core key/value tile.
__host__ __device__ constexpr int tc_block_n(int d, int dv) { return tc_paired(d, dv) ? 128 : 64; }
// Tokens per TMA store box of the paired kernel's output: one warp's 32 rows
// (32 / G tokens x G heads) when G divides 32, else the whole 128-row tile.
__host__ __device__ constexpr int out_box_tokens(int G) { return 32 % G == 0 ? 32 / G : kTcRows / G; }
// Keys per decode key/value tile for head sizes DK (K) and DV (V): a power
// of two with at most 16 KB of the wider of the two per tile.
__host__ __device__ constexpr int decode_tile_keys(int DK, int DV) {
  return (DK > DV ? DK : DV) <= 64 ? 128 : (DK > DV ? DK : DV) <= 128 ? 64 : 32;
}

// ---- workspace layout (int32 words) ----------------------------------------
// [0..8)         SchedHeader of the latest call
// [8..)          prefill order [B], prefill prefix [B+1], decode order [B],
//                decode prefix [B+1], decode completion counters [B*Hkv],
//                work counters [4]
// then (256-byte aligned) fp32 split partials [cap_units][G*dv + 2G].
// The sticky status word lives in its own allocation (it never moves when
// the workspace grows).
struct SchedHeader {
  uint32_t status;     // PVA_DEV_* bits of this call
  int32_t n_pref;      // sequences with prefill work, in pref_order
  int32_t n_items;     // prefill work items
  int32_t n_dec;       // sequences routed to split-KV decode, in dec_order
  int32_t n_units;     // decode work units (sequence, kv head, split)
  int32_t tile_tokens; // query tokens per prefill item
  int32_t units_per_tile;  // items per query tile (kv heads or heads)
  int32_t dec_chunk;   // keys per decode split
};

constexpr int kWsHeader = 0;
constexpr int kWsArrays = 8;

struct WsLayout {
  int B, Hkv;
  __host__ __device__ int pref_order() const { return kWsArrays; }
  __host__ __device__ int pref_prefix() const { return kWsArrays + B; }
  __host__ __device__ int dec_order() const { return kWsArrays + 2 * B + 1; }
  __host__ __device__ int dec_prefix() const { return kWsArrays + 3 * B + 1; }
  __host__ __device__ int dec_done() const { return kWsArrays + 4 * B + 2; }
  // work counters the persistent kernels draw item indices from: [0] prefill, [1] decode
  __host__ __device__ size_t counters() const { return (size_t)dec_done() + (size_t)B * Hkv; }
  __host__ __device__ size_t int_words() const {
    size_t w = counters() + 4;
    return (w + 63) / 64 * 64;
  }
};

// ---- per-call parameter block ------------------------------------------------
struct AttnParams {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  const int32_t* cu_q;
  const int32_t* cu_kv;
  // Optional [B]: the valid keys of each sequence, which then sits at the
  // start of its slot [cu_kv[b], cu_kv[b+1]) (padded K/V); nullptr: the whole
  // slot is the sequence.
  const int32_t* kv_len;
  // > 0: K and V are a BNSH cache [B, Hkv, kv_cap, d] (one plane of kv_cap
  // rows per (sequence, kv head)) and cu_kv[b] = b * kv_cap; 0: packed
  // [tokens, Hkv, d].
  int kv_cap;
  // > 0: K and V are padded slots [B, kv_slot, Hkv, d] read through rank-4
  // tensor maps (dims, kv heads, rows of a slot, slots), so a tile never
  // crosses into the next slot, and cu_kv[b] = b * kv_slot; 0: rank-3 maps.
  int kv_slot;
  int B, H, Hkv, G, d, dv;
  float scale;    // resolved (default already applied)
  float softcap;  // 0 = off
  int is_causal;
  int window;     // local window W > 0: keys before (causal limit + 1 - W) masked; 0 = none
  uint32_t* status;   // sticky PVA_DEV_* bits (OR-ed, cleared by pva_get_status)
  int32_t* ws;        // workspace int region
  float* partials;    // decode split partials
  int dec_cap_units;  // partial slots available
};

struct SchedConfig {
  int tile_tokens;     // query tokens per prefill item
  int units_per_tile;  // items per query tile
  int block_n;         // keys per prefill key tile (cost model only)
  int decode_enabled;  // route L_q == 1 sequences to the decode kernel
  int num_sms;
  // 1: route them there only when they are too few to fill the GPU through
  // the prefill kernel -- (L_q == 1 sequences) x kv heads < 2 x SMs --
  // because for this shape the tensor-core prefill kernel reads K/V faster
  // once it has enough (sequence, kv head) items.
  int decode_adaptive;
};

// ---- host helpers shared by the entry points (pva_api.cu) --------------------
namespace host {
// Validated launch plan of one call.
struct Plan {
  bool tensor_core = false;  // bf16/f16 tcgen05 prefill
  bool decode = false;       // split-KV decode kernel for L_q == 1
  SchedConfig sched{};
  size_t int_bytes = 0, partial_bytes = 0;
  int cap_units = 0;
};
int fail(int code, const std::string& msg);
int cuda_fail(cudaError_t e, const char* what);
int get_encoder();
int encode_map(CUtensorMap* map, const void* base, int dtype, int dim, int heads, int box_dim,
               int box_heads, int box_tokens, bool swizzle128);
// Drops pva_forward_noalloc's cached address of its static scratch on `dev`
// (the next call looks it up again in the current context).
void noalloc_forget_device(int dev);
int check_and_plan(const void* q, const void* k, const void* v, const int32_t* cu_q,
                   const int32_t* cu_kv, void* out, int B, int H, int Hkv, int d, int dv,
                   float scale, float softcap, int dtype, Plan* plan);
}  // namespace host

// Launches a kernel as a programmatic dependent of the previous work on the
// stream: it may start (and run its set-up) while that work finishes, and
// must execute griddepcontrol.wait before reading anything it produced.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// ---- launchers (defined next to their kernels) -------------------------------
cudaError_t launch_scheduler(const AttnParams& p, const SchedConfig& c, cudaStream_t s);
// One GroupQueryAttention step against a fixed-capacity BNSH KV cache (the
// front end of pva_gqa_kvcache): metadata, in-place append and rotary
// embedding, before the attention kernels read the cache.
struct CacheStep {
  const void* q;        // [B, q_seq, H, d]
  const void* k_new;    // [B, k_seq, Hkv, d]
  const void* v_new;    // [B, k_seq, Hkv, d]
  void* k_cache;        // [B, Hkv, cap, d], appended in place
  void* v_cache;
  const int32_t* seqlens_k;  // [B]: valid keys after the append, minus one
  const void* cos_cache;     // [cache_rows, rot / 2], f32 or f16
  const void* sin_cache;
  const int64_t* position_ids;  // [B, q_seq] or nullptr
  void* q_rot;          // [B, q_seq, H, d] rotated queries (rot > 0)
  int32_t* cu_q;        // [B + 1] out: b * q_seq
  int32_t* cu_kv;       // [B + 1] out: b * cap
  int32_t* kv_len;      // [B] out: total keys, or -1 (step rejected)
  int32_t* past;        // [B] out: first appended row, or -1
  int32_t* q_first;     // [B] out: position of the first query row, or -1
  uint32_t* status;
  int B, q_seq, k_seq, cap, H, Hkv, d;
  int rot, cache_rows, interleaved, rot_f16, dtype;
};
cudaError_t launch_cache_front(const CacheStep& c, cudaStream_t s);

cudaError_t launch_padded_front(const int64_t* nonpad, int B, int q_seq, int kv_seq,
                                int32_t* cu_q, int32_t* cu_kv, int32_t* kv_len, cudaStream_t s);
cudaError_t launch_prefill_f32(const AttnParams& p, int num_sms, cudaStream_t s);
cudaError_t launch_prefill_tc(const AttnParams& p, int dtype, const CUtensorMap& tq,
                              const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& to, int num_sms, cudaStream_t s);
// `to`: the output as [tokens, H, dv] with a {64, G, 128/G} box (epilogue
// stores of whole query tiles).
cudaError_t launch_prefill_pair(const AttnParams& p, int dtype, const CUtensorMap& tq,
                                const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& to, int num_sms, cudaStream_t s);
cudaError_t launch_wait_selftest(uint32_t* status, uint64_t limit_ns, int* done, cudaStream_t s);
cudaError_t launch_decode(const AttnParams& p, int dtype, const CUtensorMap& tk,
                          const CUtensorMap& tv, int num_sms, cudaStream_t s);

}  // namespace pva
