// fwd_d512.cu - prefill forward, head dim 512 (long-context workload), f16/bf16.
//
// Same online-softmax recurrence as the D = 64 kernel (attnax Pallas kernel
// body, base-2 arithmetic), reshaped for a 512-wide head:
//   * a 128 x 512 f32 accumulator alone would fill all 512 TMEM columns, so
//     each query tile is split over two CTAs, each owning 256 output columns
//     (TMEM: O half [0,256), S double buffer [256,384) and [384,512)); both
//     recompute S = Q K^T (1.5x the counted flops, still tensor-bound: per kv
//     block 2048 MMA cycles for S and 1024 for P V against ~1024 MUFU cycles
//     of softmax);
//   * Q (128 x 512, 128 KB) stays resident in shared memory as eight 64-column
//     swizzled chunks; K (eight chunks) and this CTA's half of V (four chunks)
//     stream through a 5-slot ring of 16 KB TMA chunks in the order the MMA
//     warp consumes them: K_0, then per block j: K_{j+1}, V_j;
//   * S_{j+1} is issued before P_j V, so the tensor core works on the next
//     score tile while the softmax warps work on this one;
//   * O is rescaled only when a row max grows by more than 2^8 (the running
//     max is otherwise kept stale; p <= 256 stays exact in 16-bit and the final
//     division by l cancels the common factor).
// Warp 0 TMA, warp 1 TMEM owner + MMA issue, warps 2-5 softmax (thread = row).
#include "kernels.h"

namespace attn {

constexpr int F5_NST = 5;
constexpr int F5_THREADS = 192;
constexpr uint32_t F5_CHUNK = 128 * 64 * 2;   // 16 KB: 128 rows x 64 columns
constexpr int F5_MAXKB = 2048;
constexpr float F5_RESCALE_TH = 8.f;          // log2 units

struct __align__(1024) F5Smem {
  uint8_t q[8][F5_CHUNK];
  uint8_t ring[F5_NST][F5_CHUNK];
  uint64_t full[F5_NST], empty[F5_NST];
  uint64_t qfull, sfull[2], pready, odone, alldone, fin;
  uint32_t tmem_base;
  int abort;
  int nlist;
  uint16_t list[F5_MAXKB];
  uint8_t lflags[F5_MAXKB];
};

template <bool BF16, int MOD>
__global__ void __launch_bounds__(F5_THREADS, 1) fwd_d512_kernel(const __grid_constant__ FwdBigParams p) {
  extern __shared__ uint8_t smem_raw[];
  F5Smem& sm = *reinterpret_cast<F5Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  const int L = blockIdx.x;
  const int qt = p.nqb - 1 - L / (2 * BH);   // longest causal rows first; both halves adjacent
  const int rem = L % (2 * BH);
  const int half = rem & 1;
  const int bh = rem >> 1;
  const int b = bh / p.H, h = bh % p.H;

  if (tid == 0) {
    for (int s = 0; s < F5_NST; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    mbar_init(smem_u32(&sm.qfull), 1);
    mbar_init(smem_u32(&sm.sfull[0]), 1);
    mbar_init(smem_u32(&sm.sfull[1]), 1);
    mbar_init(smem_u32(&sm.pready), 128);
    mbar_init(smem_u32(&sm.odone), 1);
    mbar_init(smem_u32(&sm.alldone), 1);
    mbar_init(smem_u32(&sm.fin), 1);
    sm.abort = 0;
    int n = 0;
    for (int kb = 0; kb < p.nkb; ++kb) {
      const int st = p.bm_tiles ? p.bm_tiles[b * p.bm_sb + h * p.bm_sh + (long long)qt * p.nkb + kb] : TILE_FULL;
      const int ks = p.km_sum ? p.km_sum[b * p.nkb + kb] : 2;   // key-padding summary of the block
      const bool visit = st != TILE_EMPTY && ks != 0;
      if (p.visited && half == 0) p.visited[((size_t)bh * p.nqb + qt) * p.nkb + kb] = visit ? 1 : 0;
      if (!visit) continue;
      sm.list[n] = (uint16_t)kb;
      sm.lflags[n] = ((st == TILE_PARTIAL && p.bm_mod != MASKMOD_NONE) ? KB_MASKMOD : 0) | (ks == 1 ? KB_KEYMASK : 0);
      ++n;
    }
    sm.nlist = n;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  const int N = sm.nlist;
  constexpr uint32_t C_O = 0, C_S = 256;

  if (warp == 0) {
    if (lane == 0 && N > 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 31};
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      const uint32_t qbar = smem_u32(&sm.qfull);
      mbar_expect_tx(qbar, 8 * F5_CHUNK);
      for (int cc = 0; cc < 8; ++cc) tma_load_2d(smem_u32(sm.q[cc]), &p.tm_q, qbar, 64 * cc, bh * p.Sq + qt * 128);
      int last_u[F5_NST];
      for (int s = 0; s < F5_NST; ++s) last_u[s] = -1;
      int u = 0;
      bool ok = true;
      // one chunk into the ring: K chunk (col = 64 cc) or this half's V chunk
      auto put = [&](const CUtensorMap* m, int col, int row) -> bool {
        const int s = u % F5_NST;
        if (u >= F5_NST && !wait_one(smem_u32(&sm.empty[s]), ((u / F5_NST) - 1) & 1, c)) return false;
        const uint32_t fb = smem_u32(&sm.full[s]);
        mbar_expect_tx(fb, F5_CHUNK);
        tma_load_2d(smem_u32(sm.ring[s]), m, fb, col, row);
        last_u[s] = u;
        ++u;
        return true;
      };
      const int krow0 = bh * p.Skv;
      for (int cc = 0; cc < 8 && ok; ++cc) ok = put(&p.tm_k, 64 * cc, krow0 + sm.list[0] * 128);
      for (int j = 0; j < N && ok; ++j) {
        if (j + 1 < N)
          for (int cc = 0; cc < 8 && ok; ++cc) ok = put(&p.tm_k, 64 * cc, krow0 + sm.list[j + 1] * 128);
        for (int cc = 0; cc < 4 && ok; ++cc) ok = put(&p.tm_v, 256 * half + 64 * cc, krow0 + sm.list[j] * 128);
      }
      {   // every copy issued has landed before the CTA exits (instant unless aborted)
        drain_wait(qbar, 0, p.timeout_ns);
        for (int s = 0; s < F5_NST; ++s)
          if (last_u[s] >= 0) drain_wait(smem_u32(&sm.full[s]), (last_u[s] / F5_NST) & 1, p.timeout_ns);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && N > 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 32};
      constexpr uint32_t ID_S = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t ID_PV = idesc_f16(128, 64, BF16, false, true);
      int u = 0;
      bool ok = wait_one(smem_u32(&sm.qfull), 0, c);
      auto issue_s = [&](int j) -> bool {
        const uint32_t d = tmem + C_S + 128 * (j & 1);
        for (int cc = 0; cc < 8; ++cc) {
          const int s = u % F5_NST;
          if (!wait_one(smem_u32(&sm.full[s]), (u / F5_NST) & 1, c)) return false;
          tc_fence_after();
          const uint32_t qa = smem_u32(sm.q[cc]), kb = smem_u32(sm.ring[s]);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)
            mma_ss(d, sdesc_sw128(qa + 32 * kk, 16, 1024), sdesc_sw128(kb + 32 * kk, 16, 1024), ID_S,
                   (cc > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&sm.empty[s]));
          ++u;
        }
        tc_commit(smem_u32(&sm.sfull[j & 1]));
        return true;
      };
      auto issue_pv = [&](int j) -> bool {
        if (!wait_one(smem_u32(&sm.pready), j & 1, c)) return false;
        tc_fence_after();
        const uint32_t a = tmem + C_S + 128 * (j & 1);
        for (int cc = 0; cc < 4; ++cc) {
          const int s = u % F5_NST;
          if (!wait_one(smem_u32(&sm.full[s]), (u / F5_NST) & 1, c)) return false;
          tc_fence_after();
          const uint32_t vb = smem_u32(sm.ring[s]);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tmem + C_O + 64 * cc, a + 8 * kk, sdesc_sw128(vb + 2048 * kk, 8192, 1024), ID_PV,
                   (j > 0 || kk > 0) ? 1u : 0u);
          tc_commit(smem_u32(&sm.empty[s]));
          ++u;
        }
        tc_commit(smem_u32(&sm.odone));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < N; ++j) {
        if (j + 1 < N && !issue_s(j + 1)) { ok = false; break; }
        if (!issue_pv(j)) { ok = false; break; }
      }
      if (ok) tc_commit(smem_u32(&sm.alldone));
      tc_commit(smem_u32(&sm.fin));
      drain_wait(smem_u32(&sm.fin), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    const int quad = warp & 3;
    const int row = 32 * quad + lane;
    const int q = qt * 128 + row;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    WaitCtx c{&sm.abort, p.status, p.timeout_ns, 33};
    const float sc = p.sc;
    float slope2 = 0.f, cb_even = 0.f;
    if constexpr (MOD == MOD_ALIBI) slope2 = alibi_slope_log2(h, p.H);
    if constexpr (MOD == MOD_CHECKER) cb_even = (q & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < N; ++j) {
      const int kv0 = sm.list[j] * 128;
      const bool causal = (MOD == MOD_CAUSAL) || ((sm.lflags[j] & KB_MASKMOD) && p.bm_mod == MASKMOD_CAUSAL);
      const int lim = q - kv0;
      if (!wait_warp(smem_u32(&sm.sfull[j & 1]), (j >> 1) & 1, c)) { ok = false; break; }
      tc_fence_after();
      const uint32_t tS = tmem + lane_off + C_S + 128 * (j & 1);
      float s[128];
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        uint32_t r[32];
        tmem_ld32(tS + 32 * jj, r);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 * jj + i] = __uint_as_float(r[i]);
      }
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
      // one straight-line copy of the pass for blocks that mix kept and padded
      // keys (a bit test per score) and one for the rest
      auto pass = [&](auto keymask_c, uint4 kw) {
        constexpr bool KM = decltype(keymask_c)::value;
#pragma unroll
        for (int cc = 0; cc < 128; ++cc) {
          float x;
          if constexpr (MOD == MOD_ALIBI)
            x = fmaf(s[cc], sc, slope2 * float(kv0 - q + cc));
          else if constexpr (MOD == MOD_CHECKER)
            x = fmaf(s[cc], sc, (cc & 1) ? -cb_even : cb_even);
          else
            x = s[cc] * sc;
          if (causal && cc > lim) x = -INFINITY;
          if constexpr (KM) {
            const uint32_t w = cc < 32 ? kw.x : (cc < 64 ? kw.y : (cc < 96 ? kw.z : kw.w));
            if (!(w & (1u << (cc & 31)))) x = -INFINITY;
          }
          s[cc] = x;
          mx[cc & 7] = fmaxf(mx[cc & 7], x);
        }
      };
      if (sm.lflags[j] & KB_KEYMASK) {
        const uint4 kw = make_uint4(km_word(p.km_bits, b, p.Skv, kv0), km_word(p.km_bits, b, p.Skv, kv0 + 32),
                                    km_word(p.km_bits, b, p.Skv, kv0 + 64), km_word(p.km_bits, b, p.Skv, kv0 + 96));
        pass(bconst<true>{}, kw);
      } else {
        pass(bconst<false>{}, make_uint4(0u, 0u, 0u, 0u));
      }
      const float rowmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                 fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      // keep a stale running max unless the new one exceeds it by 2^8
      float alpha = 1.f;
      bool resc = false;
      if (m_run == -INFINITY) {
        m_run = rowmax;                       // O holds only zeros so far: nothing to rescale
      } else if (rowmax > m_run + F5_RESCALE_TH) {
        alpha = ex2(m_run - rowmax);
        m_run = rowmax;
        resc = true;
      }
      const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
      float sum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int jj = 0; jj < 2; ++jj) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2(s[64 * jj + 2 * i] - m_use);
          const float p1 = ex2(s[64 * jj + 2 * i + 1] - m_use);
          sum[i & 3] += p0 + p1;
          pk[i] = pack2<BF16>(p0, p1);
        }
        tmem_st32(tS + 32 * jj, pk);
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold P_{j-1} V before it is rescaled (phase j-1 of odone; j >= 1 here)
        if (!wait_warp(smem_u32(&sm.odone), (j - 1) & 1, c)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int jj = 0; jj < 8; ++jj) {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + C_O + 32 * jj, r);
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
          tmem_st32(tmem + lane_off + C_O + 32 * jj, r);
        }
      }
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.pready));
      l = l * alpha + ((sum[0] + sum[1]) + (sum[2] + sum[3]));
    }
    tmem_st_wait();
    if (ok && N > 0) {
      if (!wait_warp(smem_u32(&sm.alldone), 0, c)) ok = false;
      else tc_fence_after();
    }
    if (ok) {
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint16_t* orow = reinterpret_cast<uint16_t*>(p.out) + ((size_t)bh * p.Sq + q) * 512 + 256 * half;
#pragma unroll 1
      for (int jj = 0; jj < 8; ++jj) {
        uint32_t r[32], o[16];
        if (N > 0) {
          tmem_ld32(tmem + lane_off + C_O + 32 * jj, r);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) r[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 16; ++i)
          o[i] = pack2<BF16>(__uint_as_float(r[2 * i]) * inv, __uint_as_float(r[2 * i + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * jj);
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
      }
      if (half == 0) {
        const float m_fin = (m_run == -INFINITY) ? 0.f : m_run;
        p.lse[(size_t)bh * p.Sq + q] = l > 0.f ? (m_fin + lg2(l)) * kLn2 : -INFINITY;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
}

template <bool BF16, int MOD>
static cudaError_t launch_f5_t(const FwdBigParams& p, cudaStream_t st) {
  auto kern = fwd_d512_kernel<BF16, MOD>;
  const size_t smem = sizeof(F5Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(2 * p.nqb * p.B * p.H);
  kern<<<grid, F5_THREADS, smem, st>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fwd_d512(const FwdBigParams& p, bool bf16, int mod, cudaStream_t st) {
  if (bf16) {
    switch (mod) {
      case MOD_NONE: return launch_f5_t<true, MOD_NONE>(p, st);
      case MOD_ALIBI: return launch_f5_t<true, MOD_ALIBI>(p, st);
      case MOD_CHECKER: return launch_f5_t<true, MOD_CHECKER>(p, st);
      default: return launch_f5_t<true, MOD_CAUSAL>(p, st);
    }
  }
  switch (mod) {
    case MOD_NONE: return launch_f5_t<false, MOD_NONE>(p, st);
    case MOD_ALIBI: return launch_f5_t<false, MOD_ALIBI>(p, st);
    case MOD_CHECKER: return launch_f5_t<false, MOD_CHECKER>(p, st);
    default: return launch_f5_t<false, MOD_CAUSAL>(p, st);
  }
}

}  // namespace attn
