// bwd_d512.cu - backward passes, head dim 512 (the long-context head size), f16/bf16.
//
// The same recompute backward as bwd_d64.cu (P = 2^(S scale log2e + bias log2e -
// lse log2e), dV = P^T dO, dP = dO V^T, dS = P o (dP - D), dQ = scale dS K,
// dK = scale dS^T Q), reshaped for a 512-wide head:
//   * a 128 x 512 f32 accumulator fills all 512 TMEM columns, and dK/dV need
//     two of them, so every output is split over four CTAs by head-dimension
//     quarters (128 columns each); each CTA recomputes the full score products
//     S (over all 512 dimensions) for its quarter: the score products cost 4x,
//     the gradient products 1x, about 2x the counted flops in all;
//   * no operand stays resident (a 128 x 512 tile is 128 KB): K, Q, V, dO and
//     the quarter columns stream as 16 KB (128 rows x 64 columns) TMA chunks
//     through one 8-slot ring, in exactly the order the MMA thread consumes
//     them;
//   * TMEM per CTA: S (then P, 16-bit, in place) [0, 128), dP (then dS, in
//     place) [128, 256), and the accumulators: dV [256, 384) and dK [384, 512)
//     in the dK/dV pass, dQ [256, 384) in the dQ pass.
// The score products and the gradient products of one block run back to back
// with the elementwise work between them (no overlap across blocks): this
// path is written for correctness at D = 512, the long-context forward is the
// shape's hot path.
// dK/dV pass: one CTA per (b, h, kv block, quarter): S^T = K Q^T, dP^T = V dO^T
// (kv rows on TMEM lanes), P^T and dS^T written over them as the A operands of
// dV_quarter += P^T dO_quarter and dK_quarter += dS^T Q_quarter.
// dQ pass: one CTA per (b, h, q block, quarter): S = Q K^T, dP = dO V^T, dS
// over S, dQ_quarter += dS K_quarter.
// Warp 0 TMA producer, warp 1 TMEM owner + MMA issue (lane 0), warps 2-5 one
// row each (TMEM lane = thread).
#include "kernels.h"

namespace attn {

constexpr int B5_NST = 8;                      // ring slots
constexpr int B5_THREADS = 192;
constexpr uint32_t B5_CHUNK = 128 * 64 * 2;    // 16 KB
constexpr int B5_MAXB = 2048;

struct __align__(1024) B5Smem {
  uint8_t ring[B5_NST][B5_CHUNK];
  uint64_t full[B5_NST], empty[B5_NST];
  uint64_t sfull, pready, done, fin;
  uint32_t tmem_base;
  int abort;
  int nlist;
  uint16_t list[B5_MAXB];
  uint8_t lflags[B5_MAXB];
};

// TMEM columns
constexpr uint32_t B5_S = 0, B5_DP = 128, B5_ACC0 = 256, B5_ACC1 = 384;

// Producer: one 16 KB chunk (128 rows from `row`, 64 columns from `col`) into the
// next ring slot.  `n` counts the chunks put so far.
DEVI bool b5_put(B5Smem& sm, const CUtensorMap* m, int col, int row, int& n, int (&last)[B5_NST], const WaitCtx& c) {
  const int s = n % B5_NST;
  if (n >= B5_NST && !wait_one(smem_u32(&sm.empty[s]), ((n / B5_NST) - 1) & 1, c)) return false;
  const uint32_t fb = smem_u32(&sm.full[s]);
  mbar_expect_tx(fb, B5_CHUNK);
  tma_load_2d(smem_u32(sm.ring[s]), m, fb, col, row);
  last[s] = n;
  ++n;
  return true;
}

// MMA thread: waits for chunk n and returns its slot.
DEVI int b5_take(B5Smem& sm, int n, const WaitCtx& c, bool& ok) {
  const int s = n % B5_NST;
  if (ok && !wait_one(smem_u32(&sm.full[s]), (n / B5_NST) & 1, c)) ok = false;
  return s;
}

// The score product of one block: D (+)= sum over the 8 chunks of A_c B_c^T
// (both 128 x 64, K-major), the chunks arriving in the order A_0, B_0, A_1, ...
DEVI void b5_score(B5Smem& sm, uint32_t d, int& n, uint32_t idesc, const WaitCtx& c, bool& ok) {
  for (int cc = 0; cc < 8 && ok; ++cc) {
    const int sa = b5_take(sm, n, c, ok);
    const int sb = b5_take(sm, n + 1, c, ok);
    if (!ok) break;
    tc_fence_after();
    const uint64_t ad = sdesc_sw128(smem_u32(sm.ring[sa]), 16, 1024);
    const uint64_t bd = sdesc_sw128(smem_u32(sm.ring[sb]), 16, 1024);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) mma_ss(d, ad + 2 * kk, bd + 2 * kk, idesc, (cc > 0 || kk > 0) ? 1u : 0u);
    tc_commit(smem_u32(&sm.empty[sa]));
    tc_commit(smem_u32(&sm.empty[sb]));
    n += 2;
  }
}

// The gradient product of one block for the CTA's quarter: acc[:, 64 j .. 64 j + 63]
// (+)= A (16-bit pairs in TMEM, 128 x 128) x B_j (the j-th 64-column chunk, rows =
// the K dimension, read MN-major), j = 0, 1.
DEVI void b5_grad(B5Smem& sm, uint32_t acc, uint32_t a, int& n, uint32_t idesc, bool first, const WaitCtx& c,
                  bool& ok) {
  for (int j = 0; j < 2 && ok; ++j) {
    const int sb = b5_take(sm, n, c, ok);
    if (!ok) break;
    tc_fence_after();
    const uint64_t bd = sdesc_sw128(smem_u32(sm.ring[sb]), 8192, 1024);
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) mma_ts(acc + 64 * j, a + 8 * kk, bd + 128 * kk, idesc, (!first || kk > 0) ? 1u : 0u);
    tc_commit(smem_u32(&sm.empty[sb]));
    ++n;
  }
}

// The mods and masks of one score (log2 units): x = s scale log2e + bias log2e + lse2.
template <int MOD>
DEVI float b5_logit(float s, float sc, float slope2, int q, int kv, float lse2, bool causal) {
  float x = fmaf(s, sc, lse2);
  if constexpr (MOD == MOD_ALIBI) x = fmaf(slope2, float(kv - q), x);
  if constexpr (MOD == MOD_CHECKER) x += ((q + kv) & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;
  return (causal && kv > q) ? -INFINITY : x;
}

// Work list of one CTA, built by one warp with ballots: the blocks j (of n) whose tile
// state is not EMPTY and whose keys are not all padding; for dK/dV the q blocks
// that see kv block `fixed`, for dQ the kv blocks that q block `fixed` sees.
DEVI void b5_list(B5Smem& sm, const BwdParams& p, int b, int h, int fixed, bool dkdv) {
  const int lane = lane_id();
  const int n = dkdv ? p.nqb : p.nkb;
  int cnt = 0;
  for (int j0 = 0; j0 < n; j0 += 32) {
    const int j = j0 + lane;
    bool keep = false;
    uint8_t fl = 0;
    if (j < n) {
      const int qb = dkdv ? j : fixed, kb = dkdv ? fixed : j;
      const int ks = p.km_sum ? p.km_sum[b * p.nkb + kb] : 2;
      const int st = p.bm_tiles ? p.bm_tiles[b * p.bm_sb + h * p.bm_sh + (long long)qb * p.nkb + kb] : TILE_FULL;
      keep = ks != 0 && st != TILE_EMPTY;
      fl = (st == TILE_PARTIAL && p.bm_mod != MASKMOD_NONE ? KB_MASKMOD : 0) | (ks == 1 ? KB_KEYMASK : 0);
    }
    const unsigned m = __ballot_sync(0xffffffffu, keep);
    if (keep) {
      const int pos = cnt + __popc(m & ((1u << lane) - 1u));
      sm.list[pos] = (uint16_t)j;
      sm.lflags[pos] = fl;
    }
    cnt += __popc(m);
  }
  if (lane == 0) sm.nlist = cnt;
}

DEVI void b5_setup(B5Smem& sm, int tid, int warp) {
  if (tid == 0) {
    for (int s = 0; s < B5_NST; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    mbar_init(smem_u32(&sm.sfull), 1);
    mbar_init(smem_u32(&sm.pready), 128);
    mbar_init(smem_u32(&sm.done), 1);
    mbar_init(smem_u32(&sm.fin), 1);
    sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
}

// ============================================================================
// dK / dV pass
// ============================================================================
template <bool BF16, int MOD>
__global__ void __launch_bounds__(B5_THREADS, 1) bwd512_dkdv_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  B5Smem& sm = *reinterpret_cast<B5Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  const int qr = blockIdx.x & 3;               // quarter of the 512 head dimensions
  const int kb = (blockIdx.x >> 2) / BH;       // low kv blocks (the most q blocks under causal) first
  const int bh = (blockIdx.x >> 2) % BH;
  const int b = bh / p.H, h = bh % p.H;
  b5_setup(sm, tid, warp);
  if (warp == 2) b5_list(sm, p, b, h, kb, true);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int N = sm.nlist;
  const int krow = bh * p.Skv + kb * 128;

  if (warp == 0) {
    if (lane == 0 && N > 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 51};
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      int n = 0, last[B5_NST];
      for (int s = 0; s < B5_NST; ++s) last[s] = -1;
      bool ok = true;
      for (int u = 0; u < N && ok; ++u) {
        const int qrow = bh * p.Sq + sm.list[u] * 128;
        for (int cc = 0; cc < 8 && ok; ++cc)
          ok = b5_put(sm, &p.tm_k, 64 * cc, krow, n, last, c) && b5_put(sm, &p.tm_q, 64 * cc, qrow, n, last, c);
        for (int cc = 0; cc < 8 && ok; ++cc)
          ok = b5_put(sm, &p.tm_v, 64 * cc, krow, n, last, c) && b5_put(sm, &p.tm_do, 64 * cc, qrow, n, last, c);
        for (int j = 0; j < 2 && ok; ++j) ok = b5_put(sm, &p.tm_do, 128 * qr + 64 * j, qrow, n, last, c);
        for (int j = 0; j < 2 && ok; ++j) ok = b5_put(sm, &p.tm_q, 128 * qr + 64 * j, qrow, n, last, c);
      }
      for (int s = 0; s < B5_NST; ++s)   // every copy issued lands before the CTA exits
        if (last[s] >= 0) drain_wait(smem_u32(&sm.full[s]), (last[s] / B5_NST) & 1, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && N > 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 52};
      constexpr uint32_t ID_SS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t ID_TS = idesc_f16(128, 64, BF16, false, true);
      int n = 0;
      bool ok = true;
      for (int u = 0; u < N && ok; ++u) {
        b5_score(sm, tmem + B5_S, n, ID_SS, c, ok);    // S^T = K Q^T
        b5_score(sm, tmem + B5_DP, n, ID_SS, c, ok);   // dP^T = V dO^T
        if (!ok) break;
        tc_commit(smem_u32(&sm.sfull));
        if (!wait_one(smem_u32(&sm.pready), u & 1, c)) { ok = false; break; }
        tc_fence_after();
        b5_grad(sm, tmem + B5_ACC0, tmem + B5_S, n, ID_TS, u == 0, c, ok);    // dV += P^T dO_quarter
        b5_grad(sm, tmem + B5_ACC1, tmem + B5_DP, n, ID_TS, u == 0, c, ok);   // dK += dS^T Q_quarter
      }
      if (ok) tc_commit(smem_u32(&sm.done));
      tc_commit(smem_u32(&sm.fin));   // every MMA issued completes before TMEM is freed
      drain_wait(smem_u32(&sm.fin), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    const int quad = warp & 3;
    const int r = 32 * quad + lane;   // kv row of the block
    const int kv = kb * 128 + r;
    const uint32_t lo = static_cast<uint32_t>(32 * quad) << 16;
    WaitCtx c{&sm.abort, p.status, p.timeout_ns, 53};
    const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
    // a padded key's rows stay confined to it (row r of each product reads row r of
    // its A operand) and the epilogue writes zeros for them
    bool my_key = true;
    if (p.km_bits) my_key = (km_word(p.km_bits, b, p.Skv, kv) >> (kv & 31)) & 1u;
    const float* lse2 = p.lse2 + (size_t)bh * p.Sq;
    const float* delta = p.delta + (size_t)bh * p.Sq;
    bool ok = true;
    for (int u = 0; u < N; ++u) {
      const int q0 = sm.list[u] * 128;
      const uint8_t f = sm.lflags[u];
      const bool causal = (MOD == MOD_CAUSAL && kb * 128 + 127 > q0) || ((f & KB_MASKMOD) && p.bm_mod == MASKMOD_CAUSAL);
      if (!wait_warp(smem_u32(&sm.sfull), u & 1, c)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int jj = 0; jj < 2; ++jj) {   // 64 query columns at a time; P and dS land over consumed columns
        uint32_t rr[64], pk[32];
        float pr[64];
        tmem_ld64(tmem + lo + B5_S + 64 * jj, rr);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int q = q0 + 64 * jj + i;
          pr[i] = ex2(b5_logit<MOD>(__uint_as_float(rr[i]), p.sc, slope2, q, kv, __ldg(lse2 + q), causal));
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) pk[i] = pack2<BF16>(pr[2 * i], pr[2 * i + 1]);
        tmem_st32(tmem + lo + B5_S + 32 * jj, pk);
        tmem_ld64(tmem + lo + B5_DP + 64 * jj, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int q = q0 + 64 * jj + 2 * i;
          const float d0 = pr[2 * i] * (__uint_as_float(rr[2 * i]) + __ldg(delta + q));
          const float d1 = pr[2 * i + 1] * (__uint_as_float(rr[2 * i + 1]) + __ldg(delta + q + 1));
          pk[i] = pack2<BF16>(d0, d1);
        }
        tmem_st32(tmem + lo + B5_DP + 32 * jj, pk);
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.pready));
    }
    if (ok && N > 0) {
      if (!wait_warp(smem_u32(&sm.done), 0, c)) ok = false;
      else tc_fence_after();
    }
    if (ok) {
      for (int g = 0; g < 2; ++g) {   // g = 0: dV, 1: dK (times scale)
        const float mul = (g == 0 ? 1.f : p.scale);
        uint16_t* row = reinterpret_cast<uint16_t*>(g == 0 ? p.dv : p.dk) + ((size_t)bh * p.Skv + kv) * 512 + 128 * qr;
#pragma unroll 1
        for (int jj = 0; jj < 4; ++jj) {
          uint32_t rr[32], o[16];
          if (N > 0) {
            tmem_ld32(tmem + lo + (g == 0 ? B5_ACC0 : B5_ACC1) + 32 * jj, rr);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) rr[i] = 0u;
          }
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float a0 = my_key ? __uint_as_float(rr[2 * i]) * mul : 0.f;
            const float a1 = my_key ? __uint_as_float(rr[2 * i + 1]) * mul : 0.f;
            o[i] = pack2<BF16>(a0, a1);
          }
          uint4* dst = reinterpret_cast<uint4*>(row + 32 * jj);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ============================================================================
// dQ pass
// ============================================================================
template <bool BF16, int MOD>
__global__ void __launch_bounds__(B5_THREADS, 1) bwd512_dq_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  B5Smem& sm = *reinterpret_cast<B5Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  const int qr = blockIdx.x & 3;
  const int qb = p.nqb - 1 - (blockIdx.x >> 2) / BH;   // longest causal rows first
  const int bh = (blockIdx.x >> 2) % BH;
  const int b = bh / p.H, h = bh % p.H;
  b5_setup(sm, tid, warp);
  if (warp == 2) b5_list(sm, p, b, h, qb, false);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int N = sm.nlist;
  const int qrow = bh * p.Sq + qb * 128;

  if (warp == 0) {
    if (lane == 0 && N > 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 54};
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_do);
      int n = 0, last[B5_NST];
      for (int s = 0; s < B5_NST; ++s) last[s] = -1;
      bool ok = true;
      for (int u = 0; u < N && ok; ++u) {
        const int krow = bh * p.Skv + sm.list[u] * 128;
        for (int cc = 0; cc < 8 && ok; ++cc)
          ok = b5_put(sm, &p.tm_q, 64 * cc, qrow, n, last, c) && b5_put(sm, &p.tm_k, 64 * cc, krow, n, last, c);
        for (int cc = 0; cc < 8 && ok; ++cc)
          ok = b5_put(sm, &p.tm_do, 64 * cc, qrow, n, last, c) && b5_put(sm, &p.tm_v, 64 * cc, krow, n, last, c);
        for (int j = 0; j < 2 && ok; ++j) ok = b5_put(sm, &p.tm_k, 128 * qr + 64 * j, krow, n, last, c);
      }
      for (int s = 0; s < B5_NST; ++s)
        if (last[s] >= 0) drain_wait(smem_u32(&sm.full[s]), (last[s] / B5_NST) & 1, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && N > 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 55};
      constexpr uint32_t ID_SS = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t ID_TS = idesc_f16(128, 64, BF16, false, true);
      int n = 0;
      bool ok = true;
      for (int u = 0; u < N && ok; ++u) {
        b5_score(sm, tmem + B5_S, n, ID_SS, c, ok);    // S = Q K^T
        b5_score(sm, tmem + B5_DP, n, ID_SS, c, ok);   // dP = dO V^T
        if (!ok) break;
        tc_commit(smem_u32(&sm.sfull));
        if (!wait_one(smem_u32(&sm.pready), u & 1, c)) { ok = false; break; }
        tc_fence_after();
        b5_grad(sm, tmem + B5_ACC0, tmem + B5_S, n, ID_TS, u == 0, c, ok);   // dQ += dS K_quarter
      }
      if (ok) tc_commit(smem_u32(&sm.done));
      tc_commit(smem_u32(&sm.fin));
      drain_wait(smem_u32(&sm.fin), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    const int quad = warp & 3;
    const int r = 32 * quad + lane;
    const int q = qb * 128 + r;
    const uint32_t lo = static_cast<uint32_t>(32 * quad) << 16;
    WaitCtx c{&sm.abort, p.status, p.timeout_ns, 56};
    const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
    const float nl2 = p.lse2[(size_t)bh * p.Sq + q];    // -lse log2(e)
    const float nd = p.delta[(size_t)bh * p.Sq + q];    // -D
    bool ok = true;
    for (int u = 0; u < N; ++u) {
      const int k0 = sm.list[u] * 128;
      const uint8_t f = sm.lflags[u];
      const bool causal = (MOD == MOD_CAUSAL && k0 + 127 > qb * 128) || ((f & KB_MASKMOD) && p.bm_mod == MASKMOD_CAUSAL);
      if (!wait_warp(smem_u32(&sm.sfull), u & 1, c)) { ok = false; break; }
      tc_fence_after();
#pragma unroll 1
      for (int jj = 0; jj < 2; ++jj) {
        uint32_t rr[64], pk[32];
        float pr[64];
        // key-padding bits of these 64 keys
        uint32_t kw0 = 0xffffffffu, kw1 = 0xffffffffu;
        if (p.km_bits && (f & KB_KEYMASK)) {
          kw0 = km_word(p.km_bits, b, p.Skv, k0 + 64 * jj);
          kw1 = km_word(p.km_bits, b, p.Skv, k0 + 64 * jj + 32);
        }
        tmem_ld64(tmem + lo + B5_S + 64 * jj, rr);
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          const int kv = k0 + 64 * jj + i;
          float x = b5_logit<MOD>(__uint_as_float(rr[i]), p.sc, slope2, q, kv, nl2, causal);
          x = (((i < 32 ? kw0 : kw1) >> (i & 31)) & 1u) ? x : -INFINITY;
          pr[i] = ex2(x);
        }
        tmem_ld64(tmem + lo + B5_DP + 64 * jj, rr);
#pragma unroll
        for (int i = 0; i < 32; ++i)
          pk[i] = pack2<BF16>(pr[2 * i] * (__uint_as_float(rr[2 * i]) + nd),
                              pr[2 * i + 1] * (__uint_as_float(rr[2 * i + 1]) + nd));
        tmem_st32(tmem + lo + B5_S + 32 * jj, pk);   // dS over consumed S columns
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.pready));
    }
    if (ok && N > 0) {
      if (!wait_warp(smem_u32(&sm.done), 0, c)) ok = false;
      else tc_fence_after();
    }
    if (ok) {
      uint16_t* row = reinterpret_cast<uint16_t*>(p.dq) + ((size_t)bh * p.Sq + q) * 512 + 128 * qr;
#pragma unroll 1
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t rr[32], o[16];
        if (N > 0) {
          tmem_ld32(tmem + lo + B5_ACC0 + 32 * jj, rr);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) rr[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = pack2<BF16>(__uint_as_float(rr[2 * i]) * p.scale, __uint_as_float(rr[2 * i + 1]) * p.scale);
        uint4* dst = reinterpret_cast<uint4*>(row + 32 * jj);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---------------------------------------------------------------------------
template <bool BF16, int MOD, bool DKDV>
static cudaError_t launch_b5_t(const BwdParams& p, cudaStream_t st) {
  auto kern = DKDV ? bwd512_dkdv_kernel<BF16, MOD> : bwd512_dq_kernel<BF16, MOD>;
  const size_t smem = sizeof(B5Smem) + 1024;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long long n = 4LL * p.B * p.H * (DKDV ? p.nkb : p.nqb);
  if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
  kern<<<(unsigned)n, B5_THREADS, smem, st>>>(p);
  return cudaGetLastError();
}

template <bool DKDV>
static cudaError_t launch_b5(const BwdParams& p, bool bf16, int mod, cudaStream_t st) {
  if (bf16) {
    switch (mod) {
      case MOD_NONE: return launch_b5_t<true, MOD_NONE, DKDV>(p, st);
      case MOD_ALIBI: return launch_b5_t<true, MOD_ALIBI, DKDV>(p, st);
      case MOD_CHECKER: return launch_b5_t<true, MOD_CHECKER, DKDV>(p, st);
      default: return launch_b5_t<true, MOD_CAUSAL, DKDV>(p, st);
    }
  }
  switch (mod) {
    case MOD_NONE: return launch_b5_t<false, MOD_NONE, DKDV>(p, st);
    case MOD_ALIBI: return launch_b5_t<false, MOD_ALIBI, DKDV>(p, st);
    case MOD_CHECKER: return launch_b5_t<false, MOD_CHECKER, DKDV>(p, st);
    default: return launch_b5_t<false, MOD_CAUSAL, DKDV>(p, st);
  }
}

cudaError_t launch_bwd512_dkdv(const BwdParams& p, bool bf16, int mod, cudaStream_t st) {
  return launch_b5<true>(p, bf16, mod, st);
}
cudaError_t launch_bwd512_dq(const BwdParams& p, bool bf16, int mod, cudaStream_t st) {
  return launch_b5<false>(p, bf16, mod, st);
}

}  // namespace attn
