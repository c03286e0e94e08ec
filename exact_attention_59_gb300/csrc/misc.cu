// misc.cu - the small bandwidth-bound kernels around the attention passes:
//   * key-mask packing: uint8 (B, Skv) -> bits (B, ceil(Skv/32)) and a per-(b,
//     kv block) summary that lets whole 128-key blocks be skipped or kept;
//   * the block-mask builder (the analogue of create_block_mask(mask_mod, B, H,
//     Sq, Skv) in the flaxattention README "Example usage");
//   * dense-mask packing: the (query, key) mask of the attnax
//     pallas_flash_attention arguments as row bits, column bits and tile states;
//   * the backward preprocess: -D_i = -sum_d dO_id O_id and -lse_i log2(e)
//     (-inf for rows with no kept key), negated so the passes use one FFMA.
#include "kernels.h"

namespace attn {

// One CTA of 128 threads per (b, kv block): 4 ballots give the block's 128 key bits.
__global__ void keymask_pack_kernel(const uint8_t* __restrict__ km, int Skv, uint32_t* __restrict__ bits,
                                    uint8_t* __restrict__ summary) {
  const int b = blockIdx.y, kb = blockIdx.x;
  const int kv = kb * 128 + threadIdx.x;
  const bool keep = kv < Skv && km[(size_t)b * Skv + kv] != 0;
  const unsigned w = __ballot_sync(0xffffffffu, keep);
  __shared__ int cnt[4];
  const int words = (Skv + 31) >> 5;
  const int wi = kb * 4 + (threadIdx.x >> 5);
  if ((threadIdx.x & 31) == 0) {
    if (wi < words) bits[(size_t)b * words + wi] = w;
    cnt[threadIdx.x >> 5] = __popc(w);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const int valid = min(128, Skv - kb * 128);
    const int c = cnt[0] + cnt[1] + cnt[2] + cnt[3];
    summary[(size_t)b * gridDim.x + kb] = c == 0 ? 0 : (c == valid ? 2 : 1);
  }
}

cudaError_t launch_keymask_pack(const uint8_t* km, int B, int Skv, uint32_t* bits, uint8_t* summary,
                                cudaStream_t st) {
  dim3 grid((Skv + 127) / 128, B);
  keymask_pack_kernel<<<grid, 128, 0, st>>>(km, Skv, bits, summary);
  return cudaGetLastError();
}

// Dense mask packing: one CTA of 256 threads per (mask, q tile, kv tile).  The
// tile's 128 x 128 bytes go to shared memory as 0/1 (rows padded to 132 bytes
// so that a warp reading one column touches 32 banks); a ballot over 32 lanes
// then gives each 32-bit word: along a row for rowbits, down a column for
// colbits.
__global__ void __launch_bounds__(256) dense_mask_pack_kernel(const uint8_t* __restrict__ mask, int Sq, int Skv,
                                                              int nqb, int nkb, uint8_t* __restrict__ tiles,
                                                              uint32_t* __restrict__ rowbits,
                                                              uint32_t* __restrict__ colbits) {
  __shared__ __align__(16) uint8_t t[128][132];
  __shared__ int kept;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const long long mi = blockIdx.x / ((long long)nqb * nkb);
  const int rem = (int)(blockIdx.x % ((long long)nqb * nkb));
  const int qb = rem / nkb, kb = rem % nkb;
  const uint8_t* src = mask + (size_t)mi * Sq * Skv;
  if (tid == 0) kept = 0;
  if ((Skv & 15) == 0 && (reinterpret_cast<uintptr_t>(mask) & 15) == 0) {
    // 16 bytes per load; Skv % 16 == 0 keeps each 16-byte group inside one row
    for (int i = tid; i < 128 * 8; i += 256) {
      const int r = i >> 3, c = (i & 7) * 16;
      const int q = qb * 128 + r, kv = kb * 128 + c;
      uint4 x = make_uint4(0u, 0u, 0u, 0u);
      if (q < Sq && kv < Skv) x = __ldg(reinterpret_cast<const uint4*>(src + (size_t)q * Skv + kv));
      uint32_t* d = reinterpret_cast<uint32_t*>(&t[r][c]);
      d[0] = __vcmpne4(x.x, 0u) & 0x01010101u;
      d[1] = __vcmpne4(x.y, 0u) & 0x01010101u;
      d[2] = __vcmpne4(x.z, 0u) & 0x01010101u;
      d[3] = __vcmpne4(x.w, 0u) & 0x01010101u;
    }
  } else {
    for (int i = tid; i < 128 * 128; i += 256) {
      const int r = i >> 7, c = i & 127;
      const int q = qb * 128 + r, kv = kb * 128 + c;
      t[r][c] = (q < Sq && kv < Skv && src[(size_t)q * Skv + kv] != 0) ? 1 : 0;
    }
  }
  __syncthreads();
  // rows: warp w packs rows 16 w .. 16 w + 15, one ballot per 32 columns
  int cnt = 0;
  for (int rr = 0; rr < 16; ++rr) {
    const int r = warp * 16 + rr, q = qb * 128 + r;
    uint32_t w4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w4[j] = __ballot_sync(0xffffffffu, t[r][32 * j + lane] != 0);
    cnt += __popc(w4[0]) + __popc(w4[1]) + __popc(w4[2]) + __popc(w4[3]);
    if (lane == 0 && q < Sq)
      *reinterpret_cast<uint4*>(rowbits + ((size_t)mi * Sq + q) * (4 * nkb) + 4 * kb) =
          make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
  // columns: warp w packs columns 16 w .. 16 w + 15, one ballot per 32 rows
  for (int cc = 0; cc < 16; ++cc) {
    const int c = warp * 16 + cc, kv = kb * 128 + c;
    uint32_t w4[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) w4[j] = __ballot_sync(0xffffffffu, t[32 * j + lane][c] != 0);
    if (lane == 0 && kv < Skv)
      *reinterpret_cast<uint4*>(colbits + ((size_t)mi * Skv + kv) * (4 * nqb) + 4 * qb) =
          make_uint4(w4[0], w4[1], w4[2], w4[3]);
  }
  if (lane == 0) atomicAdd(&kept, cnt);
  __syncthreads();
  if (tid == 0) {
    const long long valid = (long long)min(128, Sq - qb * 128) * min(128, Skv - kb * 128);
    tiles[blockIdx.x] = kept == 0 ? TILE_EMPTY : (kept == valid ? TILE_FULL : TILE_PARTIAL);
  }
}

cudaError_t launch_dense_mask_pack(const uint8_t* mask, long long nmask, int Sq, int Skv, uint8_t* tiles,
                                   uint32_t* rowbits, uint32_t* colbits, cudaStream_t st) {
  const int nqb = (Sq + 127) / 128, nkb = (Skv + 127) / 128;
  const long long grid = nmask * nqb * nkb;
  if (grid == 0) return cudaSuccess;
  dense_mask_pack_kernel<<<(unsigned)grid, 256, 0, st>>>(mask, Sq, Skv, nqb, nkb, tiles, rowbits, colbits);
  return cudaGetLastError();
}

// Tile state from the mask_mod over the tile's index ranges (exact for the
// mask_mods built: NONE keeps everything; CAUSAL keeps kv <= q).
__global__ void build_block_mask_kernel(int mask_mod, long long total, int Sq, int Skv, int bq, int bkv, int nqb,
                                        int nkb, uint8_t* __restrict__ tiles) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int kb = (int)(i % nkb);
    const int qb = (int)((i / nkb) % nqb);
    uint8_t st = TILE_FULL;
    if (mask_mod == MASKMOD_CAUSAL) {
      const long long q_lo = (long long)qb * bq, q_hi = min((long long)Sq, (long long)(qb + 1) * bq) - 1;
      const long long k_lo = (long long)kb * bkv, k_hi = min((long long)Skv, (long long)(kb + 1) * bkv) - 1;
      st = k_hi <= q_lo ? TILE_FULL : (k_lo > q_hi ? TILE_EMPTY : TILE_PARTIAL);
    }
    tiles[i] = st;
  }
}

cudaError_t launch_build_block_mask(int mask_mod, int B, int H, int Sq, int Skv, int bq, int bkv, uint8_t* tiles,
                                    cudaStream_t st) {
  const int nqb = (Sq + bq - 1) / bq, nkb = (Skv + bkv - 1) / bkv;
  const long long total = (long long)B * H * nqb * nkb;
  if (total == 0) return cudaSuccess;
  const long long blocks = std::min<long long>((total + 255) / 256, 152LL * 8);
  build_block_mask_kernel<<<(unsigned)blocks, 256, 0, st>>>(mask_mod, total, Sq, Skv, bq, bkv, nqb, nkb, tiles);
  return cudaGetLastError();
}

// delta_i = sum_d dout_id * out_id in f32; 16-byte loads, LPR lanes per row.
template <typename T>
DEVI void load8(const T* p, float (&f)[8]);
template <>
DEVI void load8<float>(const float* p, float (&f)[8]) {
  const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
  f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
struct h16 { uint16_t x; };
struct b16 { uint16_t x; };
template <>
DEVI void load8<h16>(const h16* p, float (&f)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack2<false>(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}
template <>
DEVI void load8<b16>(const b16* p, float (&f)[8]) {
  const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack2<true>(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

#ifndef ATTN_PRE_ROWS
#define ATTN_PRE_ROWS 2
#endif
constexpr int PRE_ROWS = ATTN_PRE_ROWS;   // rows per lane of the preprocess

template <typename T>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const T* __restrict__ out, const T* __restrict__ dout,
                                                             const float* __restrict__ lse, long long rows, int D,
                                                             float* __restrict__ delta, float* __restrict__ lse2,
                                                             long long part_rows, unsigned pre_blocks,
                                                             const uint8_t* __restrict__ km, int Skv,
                                                             uint32_t* __restrict__ bits, uint8_t* __restrict__ summary) {
  // Launched with programmatic dependent launch behind the forward: dout (an
  // input) is asked into L2 before the wait; out and lse (the forward's) are read
  // and everything is written only after it.
  if (blockIdx.x >= pre_blocks) {
    griddep_wait();
    // key-mask packing, fused into the same launch: 128 threads per (b, kv block)
    const int nkb = (Skv + 127) / 128, nkb2 = (nkb + 1) / 2;
    const int idx = (int)(blockIdx.x - pre_blocks);
    const int b = idx / nkb2, kb = (idx % nkb2) * 2 + (threadIdx.x >> 7);
    const int t = threadIdx.x & 127;
    const int kv = kb * 128 + t;
    const bool keep = kb < nkb && kv < Skv && km[(size_t)b * Skv + kv] != 0;
    const unsigned w = __ballot_sync(0xffffffffu, keep);
    __shared__ int cnt[8];
    const int words = (Skv + 31) >> 5;
    const int wi = kb * 4 + (t >> 5);
    if ((t & 31) == 0) {
      if (kb < nkb && wi < words) bits[(size_t)b * words + wi] = w;
      cnt[threadIdx.x >> 5] = __popc(w);
    }
    __syncthreads();
    if (t == 0 && kb < nkb) {
      const int g = (threadIdx.x >> 7) * 4;
      const int valid = min(128, Skv - kb * 128);
      const int c = cnt[g] + cnt[g + 1] + cnt[g + 2] + cnt[g + 3];
      summary[(size_t)b * nkb + kb] = c == 0 ? 0 : (c == valid ? 2 : 1);
    }
    return;
  }
  // D_i = rowsum(dO o O) and -lse log2(e): 8 elements per lane and chunk (a row
  // spans at most 32 lanes: D / 256 chunks per lane beyond D = 256),
  // PRE_ROWS rows per lane (row0 + k part_rows) so that 2 PRE_ROWS 16-byte
  // loads are in flight
  const int lpr = D / 8 < 32 ? D / 8 : 32;   // lanes per row
  const int per = D / (8 * lpr);            // 8-element chunks per lane
  const long long tid = blockIdx.x * (long long)blockDim.x + threadIdx.x;
  const long long row0 = tid / lpr;
  const int part = (int)(tid % lpr);
  if (threadIdx.x < PRE_ROWS) {   // this CTA's dout rows: [r0, r0 + n) and the same + k part_rows
    const long long r0 = (long long)blockIdx.x * blockDim.x / lpr;
    const long long r1 = r0 + threadIdx.x * part_rows;
    const long long n = min((long long)blockDim.x / lpr, rows - r1);
    if (r0 < part_rows && n > 0)
      prefetch_l2_bulk(dout + r1 * D, static_cast<uint32_t>(n * D * sizeof(T)));
  }
  griddep_wait();
  griddep_launch_dependents();   // the dK/dV pass may set up (it waits for this grid itself)
  float acc[PRE_ROWS];
#pragma unroll
  for (int k = 0; k < PRE_ROWS; ++k) acc[k] = 0.f;
  for (int j = 0; j < per; ++j) {
    float a[PRE_ROWS][8], g[PRE_ROWS][8];
    const int col = (part + j * lpr) * 8;
#pragma unroll
    for (int k = 0; k < PRE_ROWS; ++k) {
      const long long row = row0 + k * part_rows;
      if (row0 < part_rows && row < rows) {
        load8<T>(out + row * D + col, a[k]);
        load8<T>(dout + row * D + col, g[k]);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) a[k][i] = g[k][i] = 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < PRE_ROWS; ++k) {
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[k] = fmaf(a[k][i], g[k][i], acc[k]);
    }
  }
#pragma unroll
  for (int k = 0; k < PRE_ROWS; ++k) {
    for (int off = lpr / 2; off > 0; off >>= 1) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
    const long long row = row0 + k * part_rows;
    if (row0 < part_rows && row < rows && part == 0) {
      delta[row] = -acc[k];
      const float l = lse[row];
      lse2[row] = (l == -INFINITY) ? -INFINITY : -l * kLog2e;
    }
  }
}

cudaError_t launch_bwd_preprocess(const void* out, const void* dout, const float* lse, int dtype, long long rows,
                                  int D, float* delta, float* lse2, const uint8_t* km, int B, int Skv, uint32_t* bits,
                                  uint8_t* summary, cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  const long long part_rows = (rows + PRE_ROWS - 1) / PRE_ROWS;   // the distance between a lane's rows
  const long long threads = part_rows * (D / 8 < 32 ? D / 8 : 32);
  const unsigned pre_blocks = (unsigned)((threads + 255) / 256);
  const unsigned pack_blocks = km ? (unsigned)(B * (((Skv + 127) / 128 + 1) / 2)) : 0u;
  const unsigned grid = pre_blocks + pack_blocks;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == 0)
    return cudaLaunchKernelEx(&cfg, bwd_preprocess_kernel<float>, (const float*)out, (const float*)dout, lse, rows, D,
                              delta, lse2, part_rows, pre_blocks, km, Skv, bits, summary);
  if (dtype == 1)
    return cudaLaunchKernelEx(&cfg, bwd_preprocess_kernel<h16>, (const h16*)out, (const h16*)dout, lse, rows, D,
                              delta, lse2, part_rows, pre_blocks, km, Skv, bits, summary);
  return cudaLaunchKernelEx(&cfg, bwd_preprocess_kernel<b16>, (const b16*)out, (const b16*)dout, lse, rows, D, delta,
                            lse2, part_rows, pre_blocks, km, Skv, bits, summary);
}

}  // namespace attn
