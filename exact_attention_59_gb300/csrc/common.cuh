// common.cuh - definitions shared by the attention kernels and their launchers.
#pragma once

#ifndef __CUDACC_RTC__
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>
#endif

#include "ptx.cuh"

namespace attn {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// score_mod ids (same values as attn_score_mod in attn.h); MOD_USER is a
// score_mod compiled at run time: score + user_bias(b, h, q_idx, kv_idx)
constexpr int MOD_NONE = 0, MOD_ALIBI = 1, MOD_CHECKER = 2, MOD_CAUSAL = 3, MOD_USER = 4;
constexpr int MASKMOD_NONE = 0, MASKMOD_CAUSAL = 1, MASKMOD_USER = 2;
constexpr int TILE_EMPTY = 0, TILE_PARTIAL = 1, TILE_FULL = 2;

// The user's bias expression, in the variables b, h, q (the query position) and
// kv (the key position); only a run-time compilation defines ATTN_USER_BIAS_EXPR
// (and only it instantiates the MOD_USER kernels).
#ifdef ATTN_USER_BIAS_EXPR
__device__ __forceinline__ float user_bias(int b, int h, int q, int kv) { return (float)(ATTN_USER_BIAS_EXPR); }
#else
__device__ __forceinline__ float user_bias(int, int, int, int) { return 0.f; }
#endif
// The user's mask expression (a run-time compilation defines ATTN_USER_MASK_EXPR):
// nonzero = query position q attends to key position kv.
#ifdef ATTN_USER_MASK_EXPR
__device__ __forceinline__ bool user_keep(int b, int h, int q, int kv) { return (ATTN_USER_MASK_EXPR) != 0; }
#else
__device__ __forceinline__ bool user_keep(int, int, int, int) { return true; }
#endif

// A compile-time bool as a type: selects one straight-line copy of a loop.
template <bool V>
struct bconst {
  static constexpr bool value = V;
};

// Columns of the K = 16 augmented operands that ride on the score products
// (one more K = 16 step of S = Q K^T in the D = 64 kernels; see fwd_d64.cu):
//   forward and dQ pass: AUG_MOD .. AUG_MOD + 2 the ALiBi / checkerboard bias
//   (three 16-bit terms), AUG_KEY the key-padding mask (1 on the query side,
//   0 or -inf on the key side);
//   dK/dV pass: columns 0-2 hold the -lse terms, AUG_BMOD .. AUG_BMOD + 2 the
//   bias (the key-position part of ALiBi, or the checkerboard), AUG_MOD2 ..
//   AUG_MOD2 + 2 the query-position part of ALiBi.
constexpr int AUG_MOD = 0, AUG_KEY = 3;
constexpr int AUG_BMOD = 3, AUG_MOD2 = 6;

// Per-(q tile, kv block) work flags staged in shared memory by the prefill kernels.
constexpr uint8_t KB_VISIT = 1;    // the tile is computed
constexpr uint8_t KB_MASKMOD = 2;  // partial tile: evaluate the mask_mod per entry
constexpr uint8_t KB_KEYMASK = 4;  // some keys of the kv block are padding: test the key bits
constexpr uint8_t KB_DENSE = 8;    // the dense mask keeps only some pairs of the tile: test its bits

// Workspace layout (offsets in bytes; every region 256-byte aligned).
//   [0, 256)            status word (int32 at offset 0); item counter pairs of
//                       the forward, dK/dV and dQ passes (2 x uint32 each at
//                       kWsItemCounter, kWsDkdvCounter, kWsDqCounter); the rest
//                       reserved
//   key-mask bits       uint32 (B, Skv/32)         if a key mask may be given
//   key-mask summary    uint8  (B, ceil(Skv/128))  0 = no key kept, 1 = some, 2 = all
//   bwd: delta          float  (B, H, Sq)          -D_i = -rowsum(dO * O)
//   bwd: lse2           float  (B, H, Sq)          -lse * log2(e), -inf for empty rows
//   decode: partials    float  (B*H, nsplit, D + 2)
//   decode: counters    uint32 (B*H)
// Byte offsets, in the workspace's 256-byte header, of the item counter pairs
// of the forward, the dK/dV pass and the dQ pass (two uint32 each: items taken,
// CTAs finished; one pair per kernel, as the dQ pass may run beside the dK/dV
// pass's last CTAs).  Zero between calls: the last CTA of a call resets its
// pair, and the zero fill before first use starts them.
constexpr size_t kWsItemCounter = 16;
constexpr size_t kWsDkdvCounter = 24;
constexpr size_t kWsDqCounter = 32;

struct WsLayout {
  size_t status = 0, km_bits = 0, km_sum = 0, delta = 0, lse2 = 0, partial = 0, counter = 0, total = 0;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// ALiBi slope of head h (0-based) out of H, times log2(e): 2^(-8 (h+1) / H) * log2(e).
DEVI float alibi_slope_log2(int h, int H) { return exp2f(-8.0f * float(h + 1) / float(H)) * kLog2e; }

}  // namespace attn
