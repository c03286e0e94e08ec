// f32_tc.cu - float32 attention on the tensor cores (tcgen05 kind::tf32, three products).
//
// The same computation as the 16-bit kernels (the attnax Pallas kernel body's
// online softmax in base 2 for the forward; the recompute backward with
// D_i = rowsum(dO o O), dS = P o (dP - D), dQ = scale dS K, dK = scale dS^T Q,
// dV = P^T dO), for float32 inputs.  A kind::tf32 MMA reads 10-bit mantissas,
// so every contraction A B^T is done as three TF32 products,
//     A_hi B_hi^T + A_hi B_lo^T + A_lo B_hi^T,   x_hi = tf32(x), x_lo = tf32(x - x_hi)
// (the dropped A_lo B_lo^T is about 2^-22 of the product), accumulated in f32
// in TMEM: about f32 accuracy on the contractions.
// Written for correctness (the float32 workload is a 256-token case): one CTA
// of 128 threads per 128-row tile, each step waited for before the next, and
// the operand tiles written by the threads themselves (hi and lo parts,
// transposed where a product needs it) into 128-byte-swizzled K-major shared
// memory; P and dS go to TMEM as the A operands of the second products.
//   forward:  per 128-query tile, per 64-key step: S = Q K^T, softmax (the O
//             accumulator rescaled in TMEM when a row max grows), O += P V.
//   dQ pass:  per 128-query tile, per 64-key step: S = Q K^T, dP = dO V^T,
//             P and dS, dQ += dS K.
//   dK/dV:    per 128-key tile, per 64-query step: S^T = K Q^T, dP^T = V dO^T,
//             P^T and dS^T, dV += P^T dO, dK += dS^T Q.
// Tile skipping and masks as in the 16-bit kernels (block-mask states, key
// padding, the causal rule, the packed dense mask's tile states and bits), any
// Sq and Skv (partial last tiles: rows past the end are zeros in the operand
// tiles, get no weight, and are not written); every wait on an MMA is bounded.
#include "kernels.h"

namespace attn {

constexpr int F32_T = 128;     // threads: one row (TMEM lane) each
constexpr int F32_STEP = 64;   // keys per step (forward, dQ), queries per step (dK/dV)

struct __align__(1024) F32Smem {
  uint8_t t0hi[32768], t0lo[32768];   // resident 128 x 64 tile (Q, or K)
  uint8_t t1hi[32768], t1lo[32768];   // resident 128 x 64 tile (dO, or V), or unused
  uint8_t s0hi[16384], s0lo[16384];   // per-step 64 x 64 tiles
  uint8_t s1hi[16384], s1lo[16384];
  uint64_t bar;
  float colv[2][F32_STEP];            // per-step per-column values (dK/dV: -lse log2e, -D)
  uint8_t keep[F32_STEP];             // per-step key keep flags (forward, dQ)
  uint32_t tmem_base;
  int abort;
};

// TF32 value of x, rounded to nearest (the 19 bits a kind::tf32 MMA reads).
DEVI float tf32r(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Byte offset of element (r, c) of a K-major, 128-byte-swizzled tile of 32-bit
// elements with `rows` rows: K runs in chunks of 32 elements (128 bytes a row),
// a chunk holds rows x 128 bytes, and the 16-byte units of row r sit permuted
// by unit ^ (r & 7) (8-row, 1024-byte atoms).
DEVI uint32_t swz32(int r, int c, int rows) {
  return (uint32_t)((c >> 5) * rows * 128 + r * 128 + ((((c & 31) >> 2) ^ (r & 7)) << 4) + ((c & 3) << 2));
}

// A row-major (rows x 64) f32 tile from global memory into the hi / lo tiles,
// as is (element (r, c) at (r, c)) or transposed (at (c, r), the tile then has
// 64 rows and `rows` K columns); rows from `valid` on (past the end of the
// sequence) are zeros and are not read.  All 128 threads, 16-byte global loads.
DEVI void load_split(const float* g, int rows, uint8_t* hi, uint8_t* lo, bool transpose, int valid) {
  for (int i = threadIdx.x; i < rows * 16; i += F32_T) {
    const int r = i >> 4, c0 = (i & 15) * 4;
    const float4 v = r < valid ? __ldg(reinterpret_cast<const float4*>(g + (size_t)r * 64 + c0))
                               : make_float4(0.f, 0.f, 0.f, 0.f);
    const float x[4] = {v.x, v.y, v.z, v.w};
    if (!transpose) {
      float h[4], l[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        h[e] = tf32r(x[e]);
        l[e] = tf32r(x[e] - h[e]);
      }
      const uint32_t o = swz32(r, c0, rows);
      *reinterpret_cast<float4*>(hi + o) = make_float4(h[0], h[1], h[2], h[3]);
      *reinterpret_cast<float4*>(lo + o) = make_float4(l[0], l[1], l[2], l[3]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float h = tf32r(x[e]);
        const uint32_t o = swz32(c0 + e, r, 64);
        *reinterpret_cast<float*>(hi + o) = h;
        *reinterpret_cast<float*>(lo + o) = tf32r(x[e] - h);
      }
    }
  }
}

DEVI uint32_t idesc_tf32(int M, int N) {
  return (1u << 4)                                     // D format: f32
         | (2u << 7) | (2u << 10)                      // A, B format: TF32
         | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
DEVI void mma_tf32_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}
DEVI void mma_tf32_ts(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// D (+)= A B^T over K = 64, three TF32 products: A (128 rows) and B (nb rows)
// hi / lo tiles in shared memory (K-major, swizzled), one thread.
DEVI void mma3_ss(uint32_t d, const uint8_t* ahi, const uint8_t* alo, const uint8_t* bhi, const uint8_t* blo, int nb,
                  bool acc) {
  const uint32_t idesc = idesc_tf32(128, nb);
  for (int k8 = 0; k8 < 8; ++k8) {   // K steps of 8 elements (32 bytes)
    const uint32_t ao = (k8 >> 2) * 128 * 128 + (k8 & 3) * 32, bo = (k8 >> 2) * nb * 128 + (k8 & 3) * 32;
    const uint64_t dah = sdesc_sw128(smem_u32(ahi) + ao, 16, 1024), dal = sdesc_sw128(smem_u32(alo) + ao, 16, 1024);
    const uint64_t dbh = sdesc_sw128(smem_u32(bhi) + bo, 16, 1024), dbl = sdesc_sw128(smem_u32(blo) + bo, 16, 1024);
    mma_tf32_ss(d, dah, dbh, idesc, (acc || k8 > 0) ? 1u : 0u);
    mma_tf32_ss(d, dah, dbl, idesc, 1u);
    mma_tf32_ss(d, dal, dbh, idesc, 1u);
  }
}

// D (+)= A B^T over K = 64 with A (128 x 64, hi and lo) in TMEM columns and B
// (64 rows) hi / lo tiles in shared memory, three TF32 products, one thread.
DEVI void mma3_ts(uint32_t d, uint32_t ahi, uint32_t alo, const uint8_t* bhi, const uint8_t* blo, bool acc) {
  const uint32_t idesc = idesc_tf32(128, 64);
  for (int k8 = 0; k8 < 8; ++k8) {
    const uint32_t bo = (k8 >> 2) * 64 * 128 + (k8 & 3) * 32;
    const uint64_t dbh = sdesc_sw128(smem_u32(bhi) + bo, 16, 1024), dbl = sdesc_sw128(smem_u32(blo) + bo, 16, 1024);
    mma_tf32_ts(d, ahi + 8 * k8, dbh, idesc, (acc || k8 > 0) ? 1u : 0u);
    mma_tf32_ts(d, ahi + 8 * k8, dbl, idesc, 1u);
    mma_tf32_ts(d, alo + 8 * k8, dbh, idesc, 1u);
  }
}

// 64 f32 values of this thread's row into TMEM as hi and lo parts.
DEVI void tmem_put_split(uint32_t hi, uint32_t lo, const float (&x)[64]) {
  uint32_t h[64], l[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const float t = tf32r(x[i]);
    h[i] = __float_as_uint(t);
    l[i] = __float_as_uint(tf32r(x[i] - t));
  }
  tmem_st64(hi, h);
  tmem_st64(lo, l);
}

// Block-mask state of tile (qt, kb) for head (b, h), or FULL with no block mask.
DEVI int f32_tile_state(const SimtParams& p, int b, int h, int qt, int kb) {
  return p.bm_tiles ? p.bm_tiles[b * p.bm_sb + h * p.bm_sh + (long long)qt * p.nkb + kb] : TILE_FULL;
}

// Score in log2 units after scale, score_mod and the causal rule (the key mask is applied by the caller).
template <int MOD>
DEVI float f32_logit(float s, float sc, float slope2, int q, int kv, bool causal) {
  float x = s * sc;
  if constexpr (MOD == MOD_ALIBI) x = fmaf(slope2, float(kv - q), x);
  if constexpr (MOD == MOD_CHECKER) x += ((q + kv) & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;
  return (causal && kv > q) ? -INFINITY : x;
}

// One MMA-completion wait of the whole CTA (every warp waits, bounded); false =
// some warp gave up.  The verdict is made CTA-uniform, so every thread leaves
// the step loop together.
DEVI bool f32_wait(F32Smem& sm, const SimtParams& p, uint32_t& phase, int site) {
  WaitCtx c{&sm.abort, p.status, p.timeout_ns, site};
  const bool ok = wait_warp(smem_u32(&sm.bar), phase & 1, c);
  ++phase;
  tc_fence_after();
  return __syncthreads_and(ok ? 1 : 0) != 0;
}

DEVI void f32_setup(F32Smem& sm) {
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&sm.bar), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (threadIdx.x < 32) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// Makes the threads' shared-memory and TMEM writes visible to the MMA thread.
DEVI void f32_publish() {
  tmem_st_wait();
  fence_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
}

// On the way out: every MMA issued completes before TMEM is freed.  After a wait
// that gave up (`aborted`) thread 0 commits once more and waits (bounded) for that
// commit: it completes only after every MMA issued before it.
DEVI void f32_teardown(F32Smem& sm, const SimtParams& p, uint32_t phase, bool aborted) {
  if (threadIdx.x == 0 && aborted) {
    tc_commit(smem_u32(&sm.bar));
    drain_wait(smem_u32(&sm.bar), phase & 1, p.timeout_ns);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (threadIdx.x < 32) tmem_dealloc(sm.tmem_base, 512);
}

// ============================================================================
// forward
// ============================================================================
template <int MOD>
__global__ void __launch_bounds__(F32_T, 1) f32_fwd_kernel(const __grid_constant__ SimtParams p) {
  extern __shared__ uint8_t f32_raw[];
  F32Smem& sm = *reinterpret_cast<F32Smem*>((reinterpret_cast<uintptr_t>(f32_raw) + 1023) & ~uintptr_t(1023));
  const int qt = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int q = qt * 128 + tid;
  const bool q_in = q < p.Sq;   // rows past Sq (a partial last tile) are computed, not written
  f32_setup(sm);
  const uint32_t tm = sm.tmem_base, lo = static_cast<uint32_t>(32 * warp) << 16;
  constexpr uint32_t C_S = 0, C_O = 64, C_PH = 128, C_PL = 192;
  load_split(p.q + ((size_t)bh * p.Sq + qt * 128) * 64, 128, sm.t0hi, sm.t0lo, false, p.Sq - qt * 128);
  const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
  const long long dmi = (long long)b * p.dm.mb + (long long)h * p.dm.mh;   // dense-mask index of (b, h)
  float m = -INFINITY, l = 0.f;
  uint32_t phase = 0;
  int n = 0;
  bool ok = true;
  for (int kb = 0; kb < p.nkb && ok; ++kb) {
    const int st = f32_tile_state(p, b, h, qt, kb);
    const int ds = p.dm.tiles ? p.dm.tiles[(dmi * p.nqb + qt) * p.nkb + kb] : TILE_FULL;
    // keys of the block that exist and that the key mask keeps (the tile is skipped when none is)
    const int kv_t = kb * 128 + tid;
    const bool keep_t = kv_t < p.Skv && (p.key_mask ? p.key_mask[(size_t)b * p.Skv + kv_t] != 0 : true);
    const bool any = __syncthreads_or(keep_t);
    const bool visit = st != TILE_EMPTY && ds != TILE_EMPTY && any;
    if (p.visited && tid == 0) p.visited[((size_t)bh * p.nqb + qt) * p.nkb + kb] = visit ? 1 : 0;
    if (!visit) continue;
    const bool causal = MOD == MOD_CAUSAL || (st == TILE_PARTIAL && p.bm_mod == MASKMOD_CAUSAL);
    for (int half = 0; half < 2 && ok; ++half) {
      const int kv0 = kb * 128 + F32_STEP * half;
      if (kv0 >= p.Skv) break;   // a partial last block
      __syncthreads();   // the previous step's readers of keep and the tiles are done
      if (tid >= F32_STEP * half && tid < F32_STEP * (half + 1)) sm.keep[tid - F32_STEP * half] = keep_t ? 1 : 0;
      const size_t kvrow = (size_t)bh * p.Skv + kv0;
      load_split(p.k + kvrow * 64, F32_STEP, sm.s0hi, sm.s0lo, false, p.Skv - kv0);   // K: B of S = Q K^T
      load_split(p.v + kvrow * 64, F32_STEP, sm.s1hi, sm.s1lo, true, p.Skv - kv0);    // V^T: B of O += P V
      // this row's dense-mask bits for the step's 64 keys (a PARTIAL dense tile)
      uint32_t dw0 = 0xffffffffu, dw1 = 0xffffffffu;
      if (ds == TILE_PARTIAL && q_in) {
        const uint32_t* w = p.dm.rowbits + (dmi * p.Sq + q) * (4LL * p.nkb) + 4 * kb + 2 * half;
        dw0 = __ldg(w);
        dw1 = __ldg(w + 1);
      }
      f32_publish();
      if (tid == 0) {
        mma3_ss(tm + C_S, sm.t0hi, sm.t0lo, sm.s0hi, sm.s0lo, F32_STEP, false);
        tc_commit(smem_u32(&sm.bar));
      }
      if (!(ok = f32_wait(sm, p, phase, 61))) break;
      float x[64];
      {
        uint32_t r[64];
        tmem_ld64(tm + lo + C_S, r);
        float mx = -INFINITY;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float v = f32_logit<MOD>(__uint_as_float(r[c]), p.sc, slope2, q, kv0 + c, causal);
          v = (sm.keep[c] && (((c < 32 ? dw0 : dw1) >> (c & 31)) & 1u)) ? v : -INFINITY;
          x[c] = v;
          mx = fmaxf(mx, v);
        }
        const float m_new = fmaxf(m, mx);
        const float mu = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = (m == -INFINITY) ? 0.f : ex2(m - mu);
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          x[c] = ex2(x[c] - mu);
          sum += x[c];
        }
        l = l * alpha + sum;
        if (n > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {   // rescale O (its last product is done)
          uint32_t o[64];
          tmem_ld64(tm + lo + C_O, o);
#pragma unroll
          for (int c = 0; c < 64; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
          tmem_st64(tm + lo + C_O, o);
        }
        m = m_new;
      }
      tmem_put_split(tm + lo + C_PH, tm + lo + C_PL, x);
      f32_publish();
      if (tid == 0) {
        mma3_ts(tm + C_O, tm + C_PH, tm + C_PL, sm.s1hi, sm.s1lo, n > 0);
        tc_commit(smem_u32(&sm.bar));
      }
      if (!(ok = f32_wait(sm, p, phase, 62))) break;
      ++n;
    }
  }
  // the TMEM load stays warp-wide (tcgen05.ld is .sync.aligned): only the global
  // stores of rows past Sq are left out
  if (ok) {
    const float inv = l > 0.f ? 1.f / l : 0.f;
    uint32_t o[64];
    if (n > 0) {
      tmem_ld64(tm + lo + C_O, o);
    } else {
#pragma unroll
      for (int c = 0; c < 64; ++c) o[c] = 0u;
    }
    if (q_in) {
      float* orow = p.o + ((size_t)bh * p.Sq + q) * 64;
#pragma unroll
      for (int c = 0; c < 64; c += 4)
        *reinterpret_cast<float4*>(orow + c) = make_float4(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv,
                                                           __uint_as_float(o[c + 2]) * inv,
                                                           __uint_as_float(o[c + 3]) * inv);
      const float mf = (m == -INFINITY) ? 0.f : m;
      p.lse[(size_t)bh * p.Sq + q] = l > 0.f ? (mf + lg2(l)) * kLn2 : -INFINITY;
    }
  }
  f32_teardown(sm, p, phase, !ok);
}

// ============================================================================
// dQ pass
// ============================================================================
template <int MOD>
__global__ void __launch_bounds__(F32_T, 1) f32_dq_kernel(const __grid_constant__ SimtParams p) {
  extern __shared__ uint8_t f32_raw[];
  F32Smem& sm = *reinterpret_cast<F32Smem*>((reinterpret_cast<uintptr_t>(f32_raw) + 1023) & ~uintptr_t(1023));
  const int qt = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int q = qt * 128 + tid;
  const bool q_in = q < p.Sq;
  f32_setup(sm);
  const uint32_t tm = sm.tmem_base, lo = static_cast<uint32_t>(32 * warp) << 16;
  constexpr uint32_t C_S = 0, C_DP = 64, C_DSH = 128, C_DSL = 192, C_DQ = 256;
  const size_t qrow = (size_t)bh * p.Sq + qt * 128;
  load_split(p.q + qrow * 64, 128, sm.t0hi, sm.t0lo, false, p.Sq - qt * 128);
  load_split(p.dout + qrow * 64, 128, sm.t1hi, sm.t1lo, false, p.Sq - qt * 128);
  const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
  // rows past Sq get P = 0 and are not written
  const float nl2 = q_in ? p.lse2[(size_t)bh * p.Sq + q] : -INFINITY;   // -lse log2(e)
  const float nd = q_in ? p.delta[(size_t)bh * p.Sq + q] : 0.f;         // -D
  const long long dmi = (long long)b * p.dm.mb + (long long)h * p.dm.mh;
  uint32_t phase = 0;
  int n = 0;
  bool ok = true;
  for (int kb = 0; kb < p.nkb && ok; ++kb) {
    const int st = f32_tile_state(p, b, h, qt, kb);
    const int dst = p.dm.tiles ? p.dm.tiles[(dmi * p.nqb + qt) * p.nkb + kb] : TILE_FULL;
    const int kv_t = kb * 128 + tid;
    const bool keep_t = kv_t < p.Skv && (p.key_mask ? p.key_mask[(size_t)b * p.Skv + kv_t] != 0 : true);
    const bool any = __syncthreads_or(keep_t);
    if (st == TILE_EMPTY || dst == TILE_EMPTY || !any) continue;
    const bool causal = MOD == MOD_CAUSAL || (st == TILE_PARTIAL && p.bm_mod == MASKMOD_CAUSAL);
    for (int half = 0; half < 2 && ok; ++half) {
      const int kv0 = kb * 128 + F32_STEP * half;
      if (kv0 >= p.Skv) break;
      __syncthreads();
      if (tid >= F32_STEP * half && tid < F32_STEP * (half + 1)) sm.keep[tid - F32_STEP * half] = keep_t ? 1 : 0;
      const size_t kvrow = (size_t)bh * p.Skv + kv0;
      load_split(p.k + kvrow * 64, F32_STEP, sm.s0hi, sm.s0lo, false, p.Skv - kv0);   // K: B of S = Q K^T
      load_split(p.v + kvrow * 64, F32_STEP, sm.s1hi, sm.s1lo, false, p.Skv - kv0);   // V: B of dP = dO V^T
      uint32_t dw0 = 0xffffffffu, dw1 = 0xffffffffu;
      if (dst == TILE_PARTIAL && q_in) {
        const uint32_t* w = p.dm.rowbits + (dmi * p.Sq + q) * (4LL * p.nkb) + 4 * kb + 2 * half;
        dw0 = __ldg(w);
        dw1 = __ldg(w + 1);
      }
      f32_publish();
      if (tid == 0) {
        mma3_ss(tm + C_S, sm.t0hi, sm.t0lo, sm.s0hi, sm.s0lo, F32_STEP, false);
        mma3_ss(tm + C_DP, sm.t1hi, sm.t1lo, sm.s1hi, sm.s1lo, F32_STEP, false);
        tc_commit(smem_u32(&sm.bar));
      }
      if (!(ok = f32_wait(sm, p, phase, 63))) break;
      // K^T (B of dQ += dS K) replaces V, which the products above have read
      load_split(p.k + kvrow * 64, F32_STEP, sm.s1hi, sm.s1lo, true, p.Skv - kv0);
      float ds[64];
      {
        uint32_t r[64], dp[64];
        tmem_ld64(tm + lo + C_S, r);
        tmem_ld64(tm + lo + C_DP, dp);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float x = f32_logit<MOD>(__uint_as_float(r[c]), p.sc, slope2, q, kv0 + c, causal) + nl2;
          x = (sm.keep[c] && (((c < 32 ? dw0 : dw1) >> (c & 31)) & 1u)) ? x : -INFINITY;
          const float pp = ex2(x);
          ds[c] = pp * (__uint_as_float(dp[c]) + nd);
        }
      }
      tmem_put_split(tm + lo + C_DSH, tm + lo + C_DSL, ds);
      f32_publish();
      if (tid == 0) {
        mma3_ts(tm + C_DQ, tm + C_DSH, tm + C_DSL, sm.s1hi, sm.s1lo, n > 0);
        tc_commit(smem_u32(&sm.bar));
      }
      if (!(ok = f32_wait(sm, p, phase, 64))) break;
      ++n;
    }
  }
  if (ok) {   // warp-wide TMEM load; rows past Sq are not stored
    uint32_t o[64];
    if (n > 0) {
      tmem_ld64(tm + lo + C_DQ, o);
    } else {
#pragma unroll
      for (int c = 0; c < 64; ++c) o[c] = 0u;
    }
    if (q_in) {
      float* row = p.dq + ((size_t)bh * p.Sq + q) * 64;
#pragma unroll
      for (int c = 0; c < 64; c += 4)
        *reinterpret_cast<float4*>(row + c) =
            make_float4(__uint_as_float(o[c]) * p.scale, __uint_as_float(o[c + 1]) * p.scale,
                        __uint_as_float(o[c + 2]) * p.scale, __uint_as_float(o[c + 3]) * p.scale);
    }
  }
  f32_teardown(sm, p, phase, !ok);
}

// ============================================================================
// dK / dV pass
// ============================================================================
template <int MOD>
__global__ void __launch_bounds__(F32_T, 1) f32_dkdv_kernel(const __grid_constant__ SimtParams p) {
  extern __shared__ uint8_t f32_raw[];
  F32Smem& sm = *reinterpret_cast<F32Smem*>((reinterpret_cast<uintptr_t>(f32_raw) + 1023) & ~uintptr_t(1023));
  const int kb = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int kv = kb * 128 + tid;
  f32_setup(sm);
  const uint32_t tm = sm.tmem_base, lo = static_cast<uint32_t>(32 * warp) << 16;
  constexpr uint32_t C_S = 0, C_DP = 64, C_PH = 128, C_PL = 192, C_DSH = 256, C_DSL = 320, C_DV = 384, C_DK = 448;
  const size_t kvrow = (size_t)bh * p.Skv + kb * 128;
  // a padded key's dK and dV rows are zero; its P^T and dS^T rows stay confined to
  // it; rows past Skv (a partial last block) are not written
  const bool kv_in = kv < p.Skv;
  const bool my_key = kv_in && (p.key_mask ? p.key_mask[(size_t)b * p.Skv + kv] != 0 : true);
  const bool any_key = __syncthreads_or(my_key);
  load_split(p.k + kvrow * 64, 128, sm.t0hi, sm.t0lo, false, p.Skv - kb * 128);   // K: A of S^T = K Q^T
  load_split(p.v + kvrow * 64, 128, sm.t1hi, sm.t1lo, false, p.Skv - kb * 128);   // V: A of dP^T = V dO^T
  const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
  const long long dmi = (long long)b * p.dm.mb + (long long)h * p.dm.mh;
  uint32_t phase = 0;
  int n = 0;
  bool ok = true;
  for (int qt = 0; qt < p.nqb && ok && any_key; ++qt) {
    const int st = f32_tile_state(p, b, h, qt, kb);
    const int dst = p.dm.tiles ? p.dm.tiles[(dmi * p.nqb + qt) * p.nkb + kb] : TILE_FULL;
    if (st == TILE_EMPTY || dst == TILE_EMPTY) continue;
    const bool causal = MOD == MOD_CAUSAL || (st == TILE_PARTIAL && p.bm_mod == MASKMOD_CAUSAL);
    for (int half = 0; half < 2 && ok; ++half) {
      const int q0 = qt * 128 + F32_STEP * half;
      if (q0 >= p.Sq) break;   // a partial last q tile
      const size_t qrow = (size_t)bh * p.Sq + q0;
      __syncthreads();
      if (tid < F32_STEP) {   // queries past Sq get P = 0
        const bool in = q0 + tid < p.Sq;
        sm.colv[0][tid] = in ? p.lse2[qrow + tid] : -INFINITY;   // -lse log2(e)
        sm.colv[1][tid] = in ? p.delta[qrow + tid] : 0.f;        // -D
      }
      load_split(p.q + qrow * 64, F32_STEP, sm.s0hi, sm.s0lo, false, p.Sq - q0);      // Q: B of S^T
      load_split(p.dout + qrow * 64, F32_STEP, sm.s1hi, sm.s1lo, false, p.Sq - q0);   // dO: B of dP^T
      // this key's dense-mask bits for the step's 64 queries (a PARTIAL dense tile)
      uint32_t dw0 = 0xffffffffu, dw1 = 0xffffffffu;
      if (dst == TILE_PARTIAL && kv_in) {
        const uint32_t* w = p.dm.colbits + (dmi * p.Skv + kv) * (4LL * p.nqb) + 4 * qt + 2 * half;
        dw0 = __ldg(w);
        dw1 = __ldg(w + 1);
      }
      f32_publish();
      if (tid == 0) {
        mma3_ss(tm + C_S, sm.t0hi, sm.t0lo, sm.s0hi, sm.s0lo, F32_STEP, false);
        mma3_ss(tm + C_DP, sm.t1hi, sm.t1lo, sm.s1hi, sm.s1lo, F32_STEP, false);
        tc_commit(smem_u32(&sm.bar));
      }
      if (!(ok = f32_wait(sm, p, phase, 65))) break;
      // dO^T and Q^T (B of dV += P^T dO and dK += dS^T Q) replace Q and dO, which are read
      load_split(p.dout + qrow * 64, F32_STEP, sm.s0hi, sm.s0lo, true, p.Sq - q0);
      load_split(p.q + qrow * 64, F32_STEP, sm.s1hi, sm.s1lo, true, p.Sq - q0);
      float pr[64], ds[64];
      {
        uint32_t r[64], dp[64];
        tmem_ld64(tm + lo + C_S, r);
        tmem_ld64(tm + lo + C_DP, dp);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float x = f32_logit<MOD>(__uint_as_float(r[c]), p.sc, slope2, q0 + c, kv, causal) + sm.colv[0][c];
          x = (((c < 32 ? dw0 : dw1) >> (c & 31)) & 1u) ? x : -INFINITY;
          pr[c] = ex2(x);
          ds[c] = pr[c] * (__uint_as_float(dp[c]) + sm.colv[1][c]);
        }
      }
      tmem_put_split(tm + lo + C_PH, tm + lo + C_PL, pr);
      tmem_put_split(tm + lo + C_DSH, tm + lo + C_DSL, ds);
      f32_publish();
      if (tid == 0) {
        mma3_ts(tm + C_DV, tm + C_PH, tm + C_PL, sm.s0hi, sm.s0lo, n > 0);
        mma3_ts(tm + C_DK, tm + C_DSH, tm + C_DSL, sm.s1hi, sm.s1lo, n > 0);
        tc_commit(smem_u32(&sm.bar));
      }
      if (!(ok = f32_wait(sm, p, phase, 66))) break;
      ++n;
    }
  }
  if (ok) {   // warp-wide TMEM loads; rows past Skv are not stored
    for (int g = 0; g < 2; ++g) {   // g = 0: dV, 1: dK (times scale)
      const float mul = (g == 0 ? 1.f : p.scale) * (my_key ? 1.f : 0.f);
      float* row = (g == 0 ? p.dv : p.dk) + ((size_t)bh * p.Skv + kv) * 64;
      uint32_t o[64];
      if (n > 0) {
        tmem_ld64(tm + lo + (g == 0 ? C_DV : C_DK), o);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) o[c] = 0u;
      }
      if (!kv_in) continue;
#pragma unroll
      for (int c = 0; c < 64; c += 4) {
        float4 w;
        w.x = my_key ? __uint_as_float(o[c]) * mul : 0.f;
        w.y = my_key ? __uint_as_float(o[c + 1]) * mul : 0.f;
        w.z = my_key ? __uint_as_float(o[c + 2]) * mul : 0.f;
        w.w = my_key ? __uint_as_float(o[c + 3]) * mul : 0.f;
        *reinterpret_cast<float4*>(row + c) = w;
      }
    }
  }
  f32_teardown(sm, p, phase, !ok);
}

// ---------------------------------------------------------------------------
template <typename K>
static cudaError_t launch_f32(K kern, dim3 grid, const SimtParams& p, cudaStream_t st) {
  const size_t smem = sizeof(F32Smem) + 1024;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, F32_T, smem, st>>>(p);
  return cudaGetLastError();
}

#define ATTN_F32_DISPATCH(KERNEL, GRID)                                         \
  switch (p.mod) {                                                              \
    case MOD_NONE: return launch_f32(KERNEL<MOD_NONE>, GRID, p, st);           \
    case MOD_ALIBI: return launch_f32(KERNEL<MOD_ALIBI>, GRID, p, st);         \
    case MOD_CHECKER: return launch_f32(KERNEL<MOD_CHECKER>, GRID, p, st);     \
    default: return launch_f32(KERNEL<MOD_CAUSAL>, GRID, p, st);               \
  }

cudaError_t launch_f32_fwd(const SimtParams& p, cudaStream_t st) {
  ATTN_F32_DISPATCH(f32_fwd_kernel, dim3(p.nqb, p.B * p.H))
}
cudaError_t launch_f32_dq(const SimtParams& p, cudaStream_t st) {
  ATTN_F32_DISPATCH(f32_dq_kernel, dim3(p.nqb, p.B * p.H))
}
cudaError_t launch_f32_dkdv(const SimtParams& p, cudaStream_t st) {
  ATTN_F32_DISPATCH(f32_dkdv_kernel, dim3(p.nkb, p.B * p.H))
}
#undef ATTN_F32_DISPATCH

}  // namespace attn
