// usermask.cuh - tile states of a user mask_mod (compiled at run time, NVRTC).
//
// The analogue of create_block_mask(mask_mod, B, H, Sq, Skv) in the
// flaxattention README for a mask function given as a C expression: every
// in-range entry (q, kv) of every 128 x 128 tile of every (b, h) is evaluated
// with user_keep (common.cuh, the ATTN_USER_MASK_EXPR of the compilation); the
// tile is FULL when all of them are kept, EMPTY when none is, else PARTIAL.
// One CTA per tile at a time (grid-stride over the tiles); the CTA's verdict is
// the barrier-wide OR and AND of its threads' partial ones.
#pragma once

#include "common.cuh"

namespace attn {

constexpr int UMASK_THREADS = 256;

__global__ void __launch_bounds__(UMASK_THREADS) user_block_mask_kernel(int B, int H, int Sq, int Skv,
                                                                         uint8_t* tiles) {
  const int nqb = (Sq + 127) / 128, nkb = (Skv + 127) / 128;
  const long long ntiles = (long long)B * H * nqb * nkb;
  for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int kb = (int)(t % nkb);
    const int qb = (int)((t / nkb) % nqb);
    const long long bh = t / ((long long)nkb * nqb);
    const int b = (int)(bh / H), h = (int)(bh % H);
    const int q_hi = min(128, Sq - qb * 128), kv_hi = min(128, Skv - kb * 128);
    int any = 0, all = 1;
    for (int e = threadIdx.x; e < 128 * 128; e += UMASK_THREADS) {
      const int r = e >> 7, c = e & 127;
      if (r < q_hi && c < kv_hi) {
        const bool k = user_keep(b, h, qb * 128 + r, kb * 128 + c);
        any |= k ? 1 : 0;
        all &= k ? 1 : 0;
      }
    }
    any = __syncthreads_or(any);
    all = __syncthreads_and(all);
    if (threadIdx.x == 0) tiles[t] = all ? TILE_FULL : (any ? TILE_PARTIAL : TILE_EMPTY);
  }
}

}  // namespace attn
