// kernels.h - parameter blocks and launchers of the attention kernels.
// Included by the kernel translation units and by the C-ABI layer (api.cu).
#pragma once

#include "common.cuh"

namespace attn {

// ---------------------------------------------------------------- dense mask
// A dense (Bm, Hm, Sq, Skv) uint8 mask (Bm in {1, B}, Hm in {1, H}, nonzero =
// keep) packed once by launch_dense_mask_pack into caller memory:
//   tiles   (Bm, Hm, nqb, nkb) uint8: TILE_EMPTY (no kept pair), TILE_PARTIAL,
//           TILE_FULL (every in-range pair kept)
//   rowbits (Bm, Hm, Sq, 4 nkb) u32: bit j of word 4 kb + w = pair (q, 128 kb + 32 w + j)
//   colbits (Bm, Hm, Skv, 4 nqb) u32: bit j of word 4 qb + w = pair (128 qb + 32 w + j, kv)
// Bits of positions past Sq or Skv are 0.  Head (b, h) uses mask index
// b * mb + h * mh.
struct DenseMaskLayout {
  size_t tiles, rowbits, colbits, total;   // byte offsets and size, 256-byte aligned
};
#ifndef __CUDACC_RTC__
inline DenseMaskLayout dense_mask_layout(long long nmask, int Sq, int Skv) {
  const long long nqb = (Sq + 127) / 128, nkb = (Skv + 127) / 128;
  auto up = [](size_t x) { return (x + 255) & ~size_t(255); };
  DenseMaskLayout l;
  l.tiles = 0;
  l.rowbits = up((size_t)(nmask * nqb * nkb));
  l.colbits = l.rowbits + up((size_t)(nmask * Sq * nkb * 16));
  l.total = l.colbits + up((size_t)(nmask * Skv * nqb * 16));
  return l;
}
#endif  // host
struct DenseMaskView {
  const uint8_t* tiles;      // nullptr = no dense mask
  const uint32_t* rowbits;
  const uint32_t* colbits;
  int mb, mh;                // mask index of head (b, h) = b * mb + h * mh
};
#ifndef __CUDACC_RTC__
cudaError_t launch_dense_mask_pack(const uint8_t* mask, long long nmask, int Sq, int Skv, uint8_t* tiles,
                                   uint32_t* rowbits, uint32_t* colbits, cudaStream_t st);
#endif  // host

// ---------------------------------------------------------------- forward, D = 64
#ifndef ATTN_FWD_NST
#define ATTN_FWD_NST 3
#endif
constexpr int FWD_NST = ATTN_FWD_NST;   // forward K/V stages
constexpr int FWD_THREADS = 352;   // warp 0 TMA, warps 1-2 MMA issue (one per tile), warps 3-10 softmax
constexpr uint32_t FWD_TILE_BYTES = 128 * 64 * 2;
constexpr int FWD_MAXKB = 2048;   // Skv <= 262144

struct FwdParams {
  CUtensorMap tm_q, tm_k, tm_v;   // 2-D views (rows = B*H*S, cols = 64), box {64, 128}, 128B swizzle
  void* out;
  float* lse;
  const uint32_t* km_bits;        // (B, Skv/32) or nullptr
  const uint8_t* km_sum;          // (B, nkb) or nullptr
  // the key mask as given, bytes (B, Skv), nonzero = keep: read directly by the
  // producer (block summaries and each lane's bits) when km_bits is nullptr
  const uint8_t* km;
  const uint8_t* bm_tiles;        // block-mask states or nullptr
  long long bm_sb, bm_sh;         // element strides of b and h in bm_tiles (0 = broadcast)
  int bm_mod;
  DenseMaskView dm;               // dense (query, key) mask, dm.tiles = nullptr if none
  uint8_t* visited;               // (B, H, nqb, nkb) or nullptr
  int* status;
  int B, H, Sq, Skv, nqb, nkb, npairs;
  float sc;                       // scale * log2(e)
  unsigned long long timeout_ns;
  int inject_stall;               // test hook: the producer withholds the first K/V copy
  int q_off;                      // position of query row 0 among the keys (0 for prefill)
  // split over kv blocks: CTA split s takes blocks [s kps, (s + 1) kps) and writes
  // part (B*H, nsplit, Sq, FWD_PART) f32 rows {m (log2 units), l, 0, 0, O[64]
  // unnormalised} instead of out and lse; nsplit = 1 and part = nullptr otherwise
  int nsplit, kps;
  float* part;
  const void* kraw;               // K and V base pointers (the split variant asks L2 for its rows)
  const void* vraw;
  // Persistent CTAs: `ctas` CTAs take the items in launch order from the counter
  // items[0]; items[1] counts the CTAs that finished, and the last one resets
  // both to zero (the pair sits at a fixed workspace offset, zero before the
  // first call).  items = nullptr: one CTA per item.
  unsigned* items;
  int ctas;
  // Claims below n_whole are (query-tile pair, b, h) items; with single_tail,
  // each pair from n_whole on is claimed twice, once per query tile (the last,
  // partly filled round then runs single tiles on more CTAs).  n_whole = all
  // items without it.
  int n_whole, single_tail;
  // ALiBi / checkerboard bias folded into S = Q K^T as one more K = 16 step
  // (the AUG_MOD columns of the augmented operands), and 1 / scale
  int fold;
  float inv_scale;
};
constexpr int FWD_PART = 68;      // floats per partial row (16-byte aligned O)
#ifndef __CUDACC_RTC__
size_t fwd_d64_smem_bytes();
cudaError_t launch_fwd_d64(const FwdParams& p, bool bf16, int mod, cudaStream_t st);
cudaError_t launch_fwd_d64_kernel(const FwdParams& p, const void* kern, cudaStream_t st);
#endif  // host
// out, lse of each row from its nsplit partial rows (part as in FwdParams)
#ifndef __CUDACC_RTC__
cudaError_t launch_split_merge(const float* part, int nsplit, long long rows, int Sq, void* out, float* lse, bool bf16,
                               cudaStream_t st);
#endif  // host

// ---------------------------------------------------------------- forward, D = 512
struct FwdBigParams {
  CUtensorMap tm_q, tm_k, tm_v;   // 2-D views (rows = B*H*S, cols = 512), box {64, 128}, 128B swizzle
  void* out;
  float* lse;
  const uint32_t* km_bits;        // key mask as bits (B, ceil(Skv/32)), or nullptr
  const uint8_t* km_sum;          // (B, nkb): 0 no key kept, 1 some, 2 all
  const uint8_t* bm_tiles;
  long long bm_sb, bm_sh;
  int bm_mod;
  uint8_t* visited;
  int* status;
  int B, H, Sq, Skv, nqb, nkb;
  float sc;
  unsigned long long timeout_ns;
};
#ifndef __CUDACC_RTC__
cudaError_t launch_fwd_d512(const FwdBigParams& p, bool bf16, int mod, cudaStream_t st);
#endif  // host

// ---------------------------------------------------------------- backward, D = 64
struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;   // 2-D views, box {64, 128}, 128B swizzle
  void* dq;
  void* dk;
  void* dv;
  const float* delta;     // (B, H, Sq): -D_i = -rowsum(dO o O)
  const float* lse2;      // (B, H, Sq): -lse log2(e), -inf for rows with no kept key
  const uint32_t* km_bits;
  const uint8_t* km_sum;
  const uint8_t* bm_tiles;
  long long bm_sb, bm_sh;
  int bm_mod;
  DenseMaskView dm;
  int* status;
  int B, H, Sq, Skv, nqb, nkb;
  float sc;               // scale * log2(e)
  float scale;
  unsigned long long timeout_ns;
  int fold;               // ALiBi / checkerboard bias folded into the score products
  float inv_scale;        // 1 / scale
  // dK/dV and dQ passes, head dim 64: persistent CTAs (ctas of them) take work
  // items from the counter pair at items (items taken, CTAs finished; zero
  // between calls; one pair per pass); null: one CTA per item
  unsigned* items;
  int ctas;
};
#ifndef __CUDACC_RTC__
cudaError_t launch_bwd_dkdv(const BwdParams& p, bool bf16, int mod, cudaStream_t st);
cudaError_t launch_bwd_dq(const BwdParams& p, bool bf16, int mod, cudaStream_t st);
cudaError_t launch_bwd_kernel(const BwdParams& p, const void* kern, bool dkdv, cudaStream_t st);
// head dim 512 (f16/bf16, Sq and Skv multiples of 128; no dense mask, no user mod)
cudaError_t launch_bwd512_dkdv(const BwdParams& p, bool bf16, int mod, cudaStream_t st);
cudaError_t launch_bwd512_dq(const BwdParams& p, bool bf16, int mod, cudaStream_t st);
#endif  // host

// ---------------------------------------------------------------- small kernels
// key mask (B, Skv) uint8 -> bits (B, Skv/32) + summary (B, ceil(Skv/128))
#ifndef __CUDACC_RTC__
cudaError_t launch_keymask_pack(const uint8_t* km, int B, int Skv, uint32_t* bits, uint8_t* summary,
                                cudaStream_t st);
cudaError_t launch_build_block_mask(int mask_mod, int B, int H, int Sq, int Skv, int bq, int bkv, uint8_t* tiles,
                                    cudaStream_t st);
#endif  // host
// delta = -rowsum(dout * out) (f32), lse2 = -lse * log2(e) (-inf where lse = -inf)
// -D and -lse log2(e) per row; with km, also packs the key mask (bits + block
// summary) in the same launch.
#ifndef __CUDACC_RTC__
cudaError_t launch_bwd_preprocess(const void* out, const void* dout, const float* lse, int dtype, long long rows,
                                  int D, float* delta, float* lse2, const uint8_t* km, int B, int Skv, uint32_t* bits,
                                  uint8_t* summary, cudaStream_t st);
#endif  // host

// ---------------------------------------------------------------- decode (Sq = 1)
struct DecodeParams {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  const uint8_t* key_mask;   // (B, Skv) or nullptr
  float* partial;            // (B*H, nsplit, 2 + 64): m, l, o[64]
  unsigned* counter;         // (B*H) completion tickets (zeroed by launch_decode when used)
  int B, H, Skv, nsplit, keys_per_split;
  float sc;
  int mod;
  int cluster, ngroups;      // set by launch_decode: CTAs per cluster, clusters per (b, h),
  int rounds;                // and rounds of keys per CTA
};
#ifndef __CUDACC_RTC__
// Device-side wait limit (ATTN_TIMEOUT_NS, default 2 s), read at every call.
unsigned long long attn_timeout_ns();
int decode_num_splits(int B, int H, int Skv);
cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t st);
#endif  // host

// ---------------------------------------------------------------- f32 path (SIMT FMA)
struct SimtParams {
  const float* q;
  const float* k;
  const float* v;
  const float* out;
  const float* dout;
  float* o;
  float* lse;
  float* dq;
  float* dk;
  float* dv;
  const float* delta;
  const float* lse2;
  const uint8_t* key_mask;
  const uint8_t* bm_tiles;
  long long bm_sb, bm_sh;
  int bm_mod;
  uint8_t* visited;
  int B, H, Sq, Skv, nqb, nkb, mod;
  float sc, scale;
  int* status;                    // workspace status word (the tensor-core kernels' bounded waits)
  unsigned long long timeout_ns;
  DenseMaskView dm;               // dense (query, key) mask, dm.tiles = nullptr if none
};
#ifndef __CUDACC_RTC__
// float32 on the tensor cores (tcgen05 kind::tf32, three products per contraction)
cudaError_t launch_f32_fwd(const SimtParams& p, cudaStream_t st);
cudaError_t launch_f32_dq(const SimtParams& p, cudaStream_t st);
cudaError_t launch_f32_dkdv(const SimtParams& p, cudaStream_t st);
#endif  // host

}  // namespace attn
