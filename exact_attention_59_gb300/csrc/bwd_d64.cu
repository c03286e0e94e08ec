// bwd_d64.cu - backward passes, head dim 64, f16/bf16, tcgen05 + TMA.
//
// Gradients of sum(dO * O) (the flaxattention README differentiates
// sum(attention(...)) with jax.grad; the attnax page traces jvp through its
// forward).  Here the backward is written out, recomputing P from the saved
// lse instead of storing it (FlashAttention-2 style):
//   P = 2^(S scale log2e + bias log2e - lse log2e),  dV = P^T dO,
//   (the preprocess stores -lse log2e and -D; the dK/dV pass adds both to its
//   score products on the tensor core as one more K step, so P and dS^T cost one
//   FMUL per score; the dQ pass adds them per row, one FFMA and one
//   FADD + FMUL per pair of scores with the packed f32x2 instructions),
//   dP = dO V^T,  dS = P o (dP - D),  D_i = rowsum(dO o O),
//   dQ = scale dS K,  dK = scale dS^T Q.
// Two passes, no atomics (bitwise reproducible):
//   dK/dV pass: work items (b, h, kv block j), taken in turn by persistent CTAs
//     (one per SM) from a counter in the workspace, the next item's list, K/V
//     and first Q/dO blocks loaded under the previous item's last blocks;
//     computes S^T = K_j Q_i^T and dP^T = V_j dO_i^T directly (kv rows on TMEM
//     lanes), so P^T and dS^T are left in TMEM and feed dV += P^T dO_i and
//     dK += dS^T Q_i as the A operand.
//   dQ pass: work items (b, h, q block i), taken by persistent CTAs in the same
//     way; S = Q_i K_j^T, dP = dO_i V_j^T, dS into TMEM, dQ += dS K_j (the dQ
//     accumulator alternates between two TMEM regions from item to item).
// Both: warp 0 TMA, warp 1 TMEM owner + MMA issue (lane 0), warps 2-5 and
// 6-9 split the 128 columns of each 128x128 score tile in two halves of 64.
// S is double-buffered in TMEM so the next S product overlaps this tile's
// elementwise work.
#include "kernels.h"

namespace attn {

#ifndef ATTN_DQ_NST
#define ATTN_DQ_NST 4
#endif
constexpr int BWD_NST = ATTN_DQ_NST;   // dQ pass: K/V stages (deep enough to cover the copy latency)
#ifndef ATTN_DKDV_NST
#define ATTN_DKDV_NST 4
#endif
constexpr int DKDV_NST = ATTN_DKDV_NST;   // dK/dV pass: Q/dO stages (deep enough to cover the copy latency)
constexpr int BWD_T = 352;   // warp 0 TMA, warps 1 and 10 MMA issue, warps 2-9 elementwise
constexpr uint32_t BWD_TILE = 128 * 64 * 2;
constexpr int BWD_MAXB = 2048;

// 1-D bulk copy global -> shared, completion on an mbarrier (16-byte aligned, size % 16 == 0)
DEVI void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}


// ============================================================================
// dK / dV pass
// ============================================================================
struct __align__(1024) DkdvSmem {
  uint8_t k[BWD_TILE], v[BWD_TILE];
  uint8_t q[DKDV_NST][BWD_TILE], dO[DKDV_NST][BWD_TILE];
  // Column terms folded into the score products as one more K = 16 step:
  // qaug[s] / daug[s] hold, per q row, -lse log2(e) / (scale log2(e)) and -D
  // split as t0 + t1 + 2048 t2 (16-bit each; no swizzle, 4 KB per 128 x 16
  // operand); the key side, ones[slot], holds (1, 1, 2048) in k = 0..2 and is
  // the same in every kv row up to a period of 2, so it is 8 rows (256 bytes,
  // one per item slot) that the descriptor repeats over the 128 kv rows.  With
  // a folded ALiBi / checkerboard bias, columns AUG_BMOD.. and AUG_MOD2.. of
  // ones and of every qaug[s] carry it too (daug's stay 0).
  __align__(128) uint8_t qaug[DKDV_NST][4096];
  __align__(128) uint8_t daug[DKDV_NST][4096];
  __align__(128) uint8_t ones[2][256];
  uint64_t kvfull, kvfree, full[DKDV_NST], empty[DKDV_NST], sfull, sfree, pready, dvdone, dpfull, dpfree, dsready,
      dkdone, done, accfree, fin, finb;
  uint64_t item_ready[2], item_free[2];   // per item slot: written by the producer / done with by the rest
  uint32_t tmem_base;
  int abort;
  // Two item slots, filled by the producer in turn: the item (-1 = no more), the
  // number of q blocks that see its kv block and their list, in order, with flags.
  int item[2], nlist[2];
  uint16_t list[2][BWD_MAXB];
  uint8_t lflags[2][BWD_MAXB];
};

static_assert(sizeof(DkdvSmem) + 1024 <= 227 * 1024, "dK/dV shared memory (+ 1 KB alignment slack)");

template <bool BF16, int MOD, bool DM>
__global__ void __launch_bounds__(BWD_T, 1) bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  DkdvSmem& sm = *reinterpret_cast<DkdvSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  // Work items are (kv block, b, h), numbered so that low kv blocks come first
  // (causal: they see the most q blocks).  CTAs take them from the counter
  // p.items in turn (one CTA per SM), or, with no counter, one item each.
  const int n_items = p.nkb * BH;
  const bool persistent = p.items != nullptr;
  struct Item {
    int kb, bh, b, h;
  };
  auto item_of = [&](int L) {
    Item it;
    it.kb = L / BH;
    it.bh = L % BH;
    it.b = it.bh / p.H;
    it.h = it.bh % p.H;
    return it;
  };

  if (tid == 0) {
    mbar_init(smem_u32(&sm.kvfull), 1);
    mbar_init(smem_u32(&sm.kvfree), 1);   // thread A's commit after an item's score products
    for (int s = 0; s < DKDV_NST; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 2);   // the TMA arrival + the producer's column terms
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    mbar_init(smem_u32(&sm.sfull), 1);
    mbar_init(smem_u32(&sm.sfree), 256);
    mbar_init(smem_u32(&sm.pready), 256);
    mbar_init(smem_u32(&sm.dvdone), 1);
    mbar_init(smem_u32(&sm.dpfull), 1);
    mbar_init(smem_u32(&sm.dpfree), 256);
    mbar_init(smem_u32(&sm.dsready), 256);
    mbar_init(smem_u32(&sm.dkdone), 1);
    mbar_init(smem_u32(&sm.done), 1);
    mbar_init(smem_u32(&sm.accfree), 256);   // the elementwise threads, once dV and dK are read out
    mbar_init(smem_u32(&sm.fin), 1);
    mbar_init(smem_u32(&sm.finb), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&sm.item_ready[t]), 1);
      mbar_init(smem_u32(&sm.item_free[t]), 2 + 256);   // both MMA threads and every elementwise thread
    }
    sm.abort = 0;
    fence_mbar_init();
    fence_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  // With `fold`, the ALiBi / checkerboard bias over scale rides on S^T = K Q^T
  // (rows = keys, columns = queries), as three 16-bit terms:
  //   checkerboard  ones: (-1)^r       x  qaug: (-1)^c t_i     (t = 0.5 / scale)
  //   ALiBi         ones: t_i          x  qaug: c / 128        (t = -128 slope_h / scale)
  // r = key row of the block, c = query column of a q block (both blocks start at
  // multiples of 128, so parities are those of r and c; c / 128 is exact in both
  // 16-bit types, each product t_i c / 128 exact in f32).  ALiBi's t depends on
  // the head: the producer writes it into the item slot's ones.  ALiBi's
  // remaining slope_h (kv - q0) is one constant per kv row and q block, added
  // by the elementwise threads (thread = kv row).
  constexpr bool kModTerm = (MOD == MOD_ALIBI || MOD == MOD_CHECKER);
  const bool fold = kModTerm && p.fold;
  {
    uint4* z = reinterpret_cast<uint4*>(sm.qaug);
    for (int i = tid; i < (int)(2 * DKDV_NST * 4096 / 16); i += BWD_T) z[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < 2 * 256 / 16) reinterpret_cast<uint4*>(sm.ones)[tid] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const uint16_t one = to16<BF16>(1.f);
    if (tid < 128 && fold) {
      const int r = tid;   // a q row of the stage (query column c of S^T)
      uint16_t b3[3];
      if constexpr (MOD == MOD_CHECKER) {
        uint16_t t[3];
        split3_plain<BF16>(0.5f * p.inv_scale, t);
        for (int i = 0; i < 3; ++i) b3[i] = (r & 1) ? uint16_t(t[i] ^ 0x8000u) : t[i];
      } else {
        for (int i = 0; i < 3; ++i) b3[i] = to16<BF16>(float(r) * (1.f / 128.f));
      }
      const int col = MOD == MOD_CHECKER ? AUG_BMOD : AUG_MOD2;
      for (int st = 0; st < DKDV_NST; ++st)
        for (int i = 0; i < 3; ++i) *reinterpret_cast<uint16_t*>(sm.qaug[st] + k16_offset(r, col + i)) = b3[i];
    }
    if (tid >= 128 && tid < 128 + 16) {   // both slots' ones: 8 rows each
      const int sl = (tid - 128) >> 3, r = tid & 7;
      uint8_t* o = sm.ones[sl];
      *reinterpret_cast<uint16_t*>(o + k16_offset(r, 0)) = one;
      *reinterpret_cast<uint16_t*>(o + k16_offset(r, 1)) = one;
      *reinterpret_cast<uint16_t*>(o + k16_offset(r, 2)) = to16<BF16>(2048.f);
      if (MOD == MOD_CHECKER && fold)
        for (int i = 0; i < 3; ++i)
          *reinterpret_cast<uint16_t*>(o + k16_offset(r, AUG_BMOD + i)) = (r & 1) ? to16<BF16>(-1.f) : one;
    }
    fence_async_smem();   // generic-proxy writes, read by the tensor core
  }
  // Launched with programmatic dependent launch behind the preprocess: the set-up
  // above (barriers, TMEM, the augmented operands) reads nothing it writes; its
  // outputs (key-mask bits and summary, -lse log2(e), -D) are read only from
  // here on.  Then the dQ pass, which needs the same outputs but nothing of this
  // pass, may launch: it fills the SMs as this grid's CTAs finish.
  griddep_wait();
  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // TMEM columns: S^T 128, P^T (16-bit pairs) 64, dP^T 128, dS^T (16-bit pairs) 64, dV 64, dK 64
  constexpr uint32_t C_S = 0, C_P = 128, C_DP = 192, C_DS = 320, C_DV = 384, C_DK = 448;

  if (warp == 0) {
    // ---- producer: takes the items and fills their slots (list of q blocks, the
    // head's column term), loads an item's K and V once the previous item's score
    // products are done with them, then streams its Q / dO blocks through the
    // ring (continuing across items): lane 0 issues the TMA copies, all lanes
    // write the stage's column terms (4 q rows each), then lane 0 adds the
    // second arrival.
    WaitCtx c{&sm.abort, p.status, p.timeout_ns, 11};
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
    }
    const float inv_sc = 1.f / p.sc;
    int last_u[DKDV_NST];
    for (int s = 0; s < DKDV_NST; ++s) last_u[s] = -1;
    int u = 0, last_kv = -1;
    bool ok = true;
    for (int ci = 0; ok; ++ci) {
      const int sl = ci & 1;
      int L = 0;
      if (lane == 0) L = persistent ? (int)atomicAdd(p.items, 1u) : (ci == 0 ? (int)blockIdx.x : n_items);
      L = __shfl_sync(0xffffffffu, L, 0);
      // the slot's previous item (ci - 2) is done with everywhere
      if (ci >= 2 && !wait_warp(smem_u32(&sm.item_free[sl]), ((ci - 2) >> 1) & 1, c)) break;
      if (L >= n_items) {   // no more items: the others stop at this slot
        if (lane == 0) {
          sm.item[sl] = -1;
          mbar_arrive(smem_u32(&sm.item_ready[sl]));
        }
        break;
      }
      const Item it = item_of(L);
      // the q blocks that see this kv block, in ascending order, 32 candidates per ballot
      const int ks = p.km_sum ? p.km_sum[it.b * p.nkb + it.kb] : 2;
      int n = 0;
      if (ks != 0) {
        for (int q0 = 0; q0 < p.nqb; q0 += 32) {
          const int qb = q0 + lane;
          bool keep = false;
          uint8_t fl = 0;
          if (qb < p.nqb) {
            const int st =
                p.bm_tiles ? p.bm_tiles[it.b * p.bm_sb + it.h * p.bm_sh + (long long)qb * p.nkb + it.kb] : TILE_FULL;
            int ds = TILE_FULL;   // the dense tile state: dense build only
            if constexpr (DM)
              ds = p.dm.tiles[(((long long)it.b * p.dm.mb + (long long)it.h * p.dm.mh) * p.nqb + qb) * p.nkb + it.kb];
            keep = st != TILE_EMPTY && ds != TILE_EMPTY;
            fl = (st == TILE_PARTIAL && p.bm_mod != MASKMOD_NONE ? KB_MASKMOD : 0) | (ks == 1 ? KB_KEYMASK : 0) |
                 (ds == TILE_PARTIAL ? KB_DENSE : 0);
          }
          const unsigned m = __ballot_sync(0xffffffffu, keep);
          if (keep) {
            const int pos = n + __popc(m & ((1u << lane) - 1u));
            sm.list[sl][pos] = (uint16_t)qb;
            sm.lflags[sl][pos] = fl;
          }
          n += __popc(m);
        }
      }
      if (lane == 0) {
        sm.item[sl] = L;
        sm.nlist[sl] = n;
        if (MOD == MOD_ALIBI && fold) {
          // the head's factor of the folded -slope_h c term in the slot's ones
          // (one thread at fixed offsets: stores from every lane of the producer
          // cost the kernel registers)
          uint16_t t3[3];
          split3_plain<BF16>(-128.f * exp2f(-8.0f * float(it.h + 1) / float(p.H)) * p.inv_scale, t3);
#pragma unroll
          for (int r = 0; r < 8; ++r)
            for (int e = 0; e < 3; ++e)
              *reinterpret_cast<uint16_t*>(sm.ones[sl] + k16_offset(r, AUG_MOD2 + e)) = t3[e];
          fence_async_smem();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.item_ready[sl]));   // release: the slot is visible to its waiters
      // K and V of the item, once the previous item's score products are done with them
      if (ci >= 1 && !wait_warp(smem_u32(&sm.kvfree), (ci - 1) & 1, c)) break;
      if (lane == 0) {
        mbar_expect_tx(smem_u32(&sm.kvfull), 2 * BWD_TILE);
        tma_load_2d(smem_u32(sm.k), &p.tm_k, smem_u32(&sm.kvfull), 0, it.bh * p.Skv + it.kb * 128);
        tma_load_2d(smem_u32(sm.v), &p.tm_v, smem_u32(&sm.kvfull), 0, it.bh * p.Skv + it.kb * 128);
      }
      last_kv = ci;
      for (int j = 0; j < n; ++j) {
        const int s = u % DKDV_NST;
        if (u >= DKDV_NST && !wait_warp(smem_u32(&sm.empty[s]), ((u / DKDV_NST) - 1) & 1, c)) {
          ok = false;
          break;
        }
        const int qb = sm.list[sl][j];
        const uint32_t fb = smem_u32(&sm.full[s]);
        const int row = it.bh * p.Sq + qb * 128;
        if (lane == 0) {
          mbar_expect_tx(fb, 2 * BWD_TILE);
          tma_load_2d(smem_u32(sm.q[s]), &p.tm_q, fb, 0, row);
          tma_load_2d(smem_u32(sm.dO[s]), &p.tm_do, fb, 0, row);
        }
        float xl[4], xd[4];
        if ((p.Sq & 3) == 0 && qb * 128 + 128 <= p.Sq) {   // whole block, 16-byte aligned rows
          const float4 nl = __ldg(reinterpret_cast<const float4*>(p.lse2 + row) + lane);
          const float4 nd = __ldg(reinterpret_cast<const float4*>(p.delta + row) + lane);
          xl[0] = nl.x * inv_sc; xl[1] = nl.y * inv_sc; xl[2] = nl.z * inv_sc; xl[3] = nl.w * inv_sc;
          xd[0] = nd.x; xd[1] = nd.y; xd[2] = nd.z; xd[3] = nd.w;
        } else {   // rows past Sq (partial last q block) get P = 0: the infinity that the scale turns into -inf
          const float pad = p.sc < 0.f ? INFINITY : -INFINITY;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool in = qb * 128 + 4 * lane + i < p.Sq;
            xl[i] = in ? __ldg(p.lse2 + row + 4 * lane + i) * inv_sc : pad;
            xd[i] = in ? __ldg(p.delta + row + 4 * lane + i) : 0.f;
          }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int r = 4 * lane + i;
          split3<BF16>(xl[i], sm.qaug[s], r);
          split3<BF16>(xd[i], sm.daug[s], r);
        }
        fence_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(fb);
        last_u[s] = u;
        ++u;
      }
    }
    if (lane == 0) {   // every copy issued has landed before the CTA exits (instant unless aborted)
      if (last_kv >= 0) drain_wait(smem_u32(&sm.kvfull), last_kv & 1, p.timeout_ns);
      for (int s = 0; s < DKDV_NST; ++s)
        if (last_u[s] >= 0) drain_wait(smem_u32(&sm.full[s]), (last_u[s] / DKDV_NST) & 1, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issue, thread A: the score products S^T = K Q^T and dP^T = V dO^T.
    // S^T(u) is issued as soon as the elementwise warps hold S^T(u-1) in registers
    // and dP^T(u) as soon as they hold dP^T(u-1): P^T and dS^T live in TMEM
    // regions of their own, so the score products never wait for the gradient
    // products.  u counts blocks over all items of the CTA (the barriers' phases).
    if (lane == 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 12};
      constexpr uint32_t ID_SS = idesc_f16(128, 128, BF16, false, false);
      const uint64_t kd = sdesc_sw128(smem_u32(sm.k), 16, 1024), vd = sdesc_sw128(smem_u32(sm.v), 16, 1024);
      uint32_t u = 0;
      bool ok = true;
      for (int ci = 0; ok; ++ci) {
        const int sl = ci & 1;
        if (!wait_one(smem_u32(&sm.item_ready[sl]), (ci >> 1) & 1, c)) break;
        if (sm.item[sl] < 0) break;
        const int n = sm.nlist[sl];
        const uint64_t oned = sdesc_k16_rows8(smem_u32(sm.ones[sl]));
        if (!wait_one(smem_u32(&sm.kvfull), ci & 1, c)) break;
        for (int j = 0; j < n; ++j, ++u) {
          const int s = u % DKDV_NST;
          if (!wait_one(smem_u32(&sm.full[s]), (u / DKDV_NST) & 1, c)) { ok = false; break; }
          if (u > 0 && !wait_one(smem_u32(&sm.sfree), (u - 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
          {   // S^T_u = K Q_u^T - lse_q / scale
            const uint64_t qd = sdesc_sw128(smem_u32(sm.q[s]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + C_S, kd + 2 * kk, qd + 2 * kk, ID_SS, kk > 0);
            mma_ss(tmem + C_S, oned, sdesc_k16(smem_u32(sm.qaug[s])), ID_SS, 1u);
            tc_commit(smem_u32(&sm.sfull));
          }
          if (u > 0 && !wait_one(smem_u32(&sm.dpfree), (u - 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
          {   // dP^T_u = V dO_u^T - D_q
            const uint64_t od = sdesc_sw128(smem_u32(sm.dO[s]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + C_DP, vd + 2 * kk, od + 2 * kk, ID_SS, kk > 0);
            mma_ss(tmem + C_DP, oned, sdesc_k16(smem_u32(sm.daug[s])), ID_SS, 1u);
            tc_commit(smem_u32(&sm.dpfull));
          }
        }
        if (!ok) break;
        // both arrive once this item's score products are complete: K and V may be
        // reloaded, and the slot (its ones) refilled
        tc_commit(smem_u32(&sm.kvfree));
        tc_commit(smem_u32(&sm.item_free[sl]));
      }
      // every MMA issued by this thread completes before the CTA lets go of TMEM
      tc_commit(smem_u32(&sm.fin));
      drain_wait(smem_u32(&sm.fin), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ---- MMA issue, thread B: the gradient products dV += P^T dO and dK += dS^T Q,
    // A operands read from TMEM where the elementwise warps left P^T and dS^T.  An
    // item's first products overwrite dV and dK, once the elementwise warps have
    // read the previous item's out (accfree).
    if (lane == 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 14};
      constexpr uint32_t ID_TS = idesc_f16(128, 64, BF16, false, true);
      uint32_t u = 0;
      bool ok = true;
      for (int ci = 0; ok; ++ci) {
        const int sl = ci & 1;
        if (!wait_one(smem_u32(&sm.item_ready[sl]), (ci >> 1) & 1, c)) break;
        if (sm.item[sl] < 0) break;
        const int n = sm.nlist[sl];
        if (ci >= 1 && !wait_one(smem_u32(&sm.accfree), (ci - 1) & 1, c)) break;
        tc_fence_after();
        for (int j = 0; j < n; ++j, ++u) {
          const int s = u % DKDV_NST;
          if (!wait_one(smem_u32(&sm.full[s]), (u / DKDV_NST) & 1, c)) { ok = false; break; }
          if (!wait_one(smem_u32(&sm.pready), u & 1, c)) { ok = false; break; }
          tc_fence_after();
          {   // dV += P^T dO_u
            const uint64_t od = sdesc_sw128(smem_u32(sm.dO[s]), 8192, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C_DV, tmem + C_P + 8 * kk, od + 128 * kk, ID_TS, (j > 0 || kk > 0));
            tc_commit(smem_u32(&sm.dvdone));
          }
          if (!wait_one(smem_u32(&sm.dsready), u & 1, c)) { ok = false; break; }
          tc_fence_after();
          {   // dK += dS^T Q_u
            const uint64_t qd = sdesc_sw128(smem_u32(sm.q[s]), 8192, 1024);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma_ts(tmem + C_DK, tmem + C_DS + 8 * kk, qd + 128 * kk, ID_TS, (j > 0 || kk > 0));
            tc_commit(smem_u32(&sm.dkdone));
          }
          tc_commit(smem_u32(&sm.empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.done));   // this item's dV and dK are complete once it arrives
        mbar_arrive(smem_u32(&sm.item_free[sl]));
      }
      tc_commit(smem_u32(&sm.finb));
      drain_wait(smem_u32(&sm.finb), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    const int w = (warp - 2) >> 2;   // column half: q columns [64 w, 64 w + 64)
    const int quad = warp & 3;
    const int r = 32 * quad + lane;  // kv row in the block
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    WaitCtx c{&sm.abort, p.status, p.timeout_ns, 13 + w};
    const uint64_t scv = f2(p.sc, p.sc);
    uint32_t u = 0;   // blocks over all items (the barriers' phases)
    bool ok = true;
    for (int ci = 0; ok; ++ci) {
      const int sl = ci & 1;
      if (!wait_warp(smem_u32(&sm.item_ready[sl]), (ci >> 1) & 1, c)) break;
      const int L = sm.item[sl];
      if (L < 0) break;
      const Item it = item_of(L);
      const int kb = it.kb, bh = it.bh, b = it.b, h = it.h;
      const int N = sm.nlist[sl];
      const int kv = kb * 128 + r;
      const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
      // A padded key's dK and dV rows are zero.  Its P^T and dS^T rows are not masked
      // here: row r of an MMA result depends on row r of its A operand only, so
      // those rows stay confined to the padded key and the epilogue writes zeros.
      bool my_key = kv < p.Skv;   // rows past Skv (partial last kv block) are not written
      if (p.km_bits && my_key) my_key = (km_word(p.km_bits, b, p.Skv, kv) >> (kv & 31)) & 1u;
      for (int j = 0; j < N; ++j, ++u) {
        const int qb = sm.list[sl][j];
        const uint8_t f = sm.lflags[sl][j];
        const int q0 = qb * 128 + 64 * w;   // first query of this half
        const bool causal = (MOD == MOD_CAUSAL && kb * 128 + 127 > qb * 128) ||
                            ((f & KB_MASKMOD) && p.bm_mod == MASKMOD_CAUSAL);
        const bool umask = MOD == MOD_USER && (f & KB_MASKMOD) && p.bm_mod == MASKMOD_USER;
        // this key's dense-mask bits for the half's 64 queries (column words)
        bool dense = false;
        uint2 dwv = make_uint2(0u, 0u);
        if constexpr (DM) {
          dense = f & KB_DENSE;
          const long long dmi = (long long)b * p.dm.mb + (long long)h * p.dm.mh;
          if (dense && kv < p.Skv)
            dwv = __ldg(reinterpret_cast<const uint2*>(p.dm.colbits + (dmi * p.Skv + kv) * (4LL * p.nqb) + 4 * qb +
                                                       2 * w));
        }
        // the block's bias constants, ahead of the wait (they do not depend on S^T)
        uint64_t chk = 0;
        if constexpr (MOD == MOD_CHECKER) {
          const float hb = ((kv + q0) & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;   // even column
          chk = f2(hb, -hb);
        }
        const float abase = (MOD == MOD_ALIBI) ? slope2 * float(kv - q0) : 0.f;
        // with the bias folded into S^T, slope_h (kv - qb 128) is left: one constant per row
        const float fb = (MOD == MOD_ALIBI) ? slope2 * float(kv - qb * 128) : 0.f;
        const uint64_t fbv = f2(fb, fb);
        if (!wait_warp(smem_u32(&sm.sfull), u & 1, c)) { ok = false; break; }
        tc_fence_after();
        uint32_t rr[64];
        tmem_ld64(tmem + lane_off + C_S + 64 * w, rr);
        // S^T(u) is in registers: the next S^T may be computed over it
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.sfree));
        float pr[64];
        uint32_t pk[32];
        // one straight-line copy per causal/not: no runtime test inside the unrolled loop
        auto probs = [&](auto causal_c, auto dense_c, auto fold_c) {
          constexpr bool CAUSAL = decltype(causal_c)::value;
          constexpr bool DENSE = decltype(dense_c)::value;
          constexpr bool FOLD = decltype(fold_c)::value;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const uint64_t sv = f2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1]));
            uint64_t xv = FOLD ? ffma2(sv, scv, fbv) : fmul2(sv, scv);
            if constexpr (MOD == MOD_CHECKER && !FOLD) xv = fadd2(xv, chk);
            if constexpr (MOD == MOD_ALIBI && !FOLD)
              xv = fadd2(xv, f2(fmaf(-slope2, float(2 * i), abase), fmaf(-slope2, float(2 * i + 1), abase)));
            float x0, x1;
            unf2(xv, x0, x1);
            if constexpr (MOD == MOD_USER) {
              x0 = fmaf(user_bias(b, h, q0 + 2 * i, kv), kLog2e, x0);
              x1 = fmaf(user_bias(b, h, q0 + 2 * i + 1, kv), kLog2e, x1);
              if (umask) {   // a PARTIAL tile of a user mask_mod's block mask
                x0 = user_keep(b, h, q0 + 2 * i, kv) ? x0 : -INFINITY;
                x1 = user_keep(b, h, q0 + 2 * i + 1, kv) ? x1 : -INFINITY;
              }
            }
            if (CAUSAL) {
              x0 = kv > q0 + 2 * i ? -INFINITY : x0;
              x1 = kv > q0 + 2 * i + 1 ? -INFINITY : x1;
            }
            if constexpr (DENSE) {
              const uint32_t dwi = i < 16 ? dwv.x : dwv.y;
              x0 = (dwi & (1u << ((2 * i) & 31))) ? x0 : -INFINITY;
              x1 = (dwi & (1u << ((2 * i + 1) & 31))) ? x1 : -INFINITY;
            }
            const float p0 = ex2(x0), p1 = ex2(x1);
            pr[2 * i] = p0;
            pr[2 * i + 1] = p1;
            pk[i] = pack2<BF16>(p0, p1);
          }
        };
        auto probs_any = [&](auto fold_c) {
          if (dense) {   // never with DM = false
            if constexpr (DM) {
              if (causal) probs(bconst<true>{}, bconst<true>{}, fold_c);
              else probs(bconst<false>{}, bconst<true>{}, fold_c);
            }
          } else {
            if (causal) probs(bconst<true>{}, bconst<false>{}, fold_c);
            else probs(bconst<false>{}, bconst<false>{}, fold_c);
          }
        };
        if constexpr (kModTerm) {
          if (fold) probs_any(bconst<true>{});
          else probs_any(bconst<false>{});
        } else {
          probs_any(bconst<false>{});
        }
        // dV(u-1) has finished reading the P^T region
        if (u > 0) {
          if (!wait_warp(smem_u32(&sm.dvdone), (u - 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st32(tmem + lane_off + C_P + 32 * w, pk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.pready));
        if (!wait_warp(smem_u32(&sm.dpfull), u & 1, c)) { ok = false; break; }
        tc_fence_after();
        tmem_ld64(tmem + lane_off + C_DP + 64 * w, rr);
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.dpfree));
        uint32_t dsk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const uint64_t dd = f2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1]));   // dP - D
          float d0, d1;
          unf2(fmul2(f2(pr[2 * i], pr[2 * i + 1]), dd), d0, d1);
          dsk[i] = pack2<BF16>(d0, d1);
        }
        // dK(u-1) has finished reading the dS^T region
        if (u > 0) {
          if (!wait_warp(smem_u32(&sm.dkdone), (u - 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st32(tmem + lane_off + C_DS + 32 * w, dsk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.dsready));
      }
      tmem_st_wait();
      if (!ok) break;
      // epilogue: warps 2-5 write dV rows, warps 6-9 write dK rows (scaled)
      if (!wait_warp(smem_u32(&sm.done), ci & 1, c)) break;
      tc_fence_after();
      {
        const float mul = (w == 0 ? 1.f : p.scale) * (my_key ? 1.f : 0.f);
        uint32_t rr[64], o[32];
        if (N > 0) {
          tmem_ld64(tmem + lane_off + (w == 0 ? C_DV : C_DK), rr);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) rr[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          // multiply, not select: a padded key's rows may hold any finite value
          const float a0 = my_key ? __uint_as_float(rr[2 * i]) * mul : 0.f;
          const float a1 = my_key ? __uint_as_float(rr[2 * i + 1]) * mul : 0.f;
          o[i] = pack2<BF16>(a0, a1);
        }
        uint16_t* base = reinterpret_cast<uint16_t*>(w == 0 ? p.dv : p.dk);
        uint4* dst = reinterpret_cast<uint4*>(base + ((size_t)bh * p.Skv + kv) * 64);
        if (kv < p.Skv) {
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
      // dV and dK are read out (the TMEM load above waits): the next item's first
      // products may overwrite them; and this item's slot is done with
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.accfree));
      mbar_arrive(smem_u32(&sm.item_free[sl]));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  // the last CTA to finish re-arms the item counter for the next call (this
  // thread made the CTA's last claim, so every claim precedes the reset)
  if (persistent && tid == 0) {
    __threadfence();
    if (atomicAdd(p.items + 1, 1u) == gridDim.x - 1u) {
      p.items[0] = 0u;
      p.items[1] = 0u;
    }
  }
}

// ============================================================================
// dQ pass
// ============================================================================
struct __align__(1024) DqSmem {
  uint8_t q[BWD_TILE], dO[BWD_TILE];
  uint8_t k[BWD_NST][BWD_TILE], v[BWD_NST][BWD_TILE];
  // Column terms folded into S = Q K^T as one more K = 16 step, as in the
  // forward (columns AUG_MOD / AUG_KEY; K = 16 operands without swizzle):
  // kaug[s] per key of stage s (4 KB each); the query side is the same in every
  // row up to a period of 2, so it is 8 rows (256 bytes, one per item slot) that
  // the descriptor repeats over the 128 query rows.
  __align__(128) uint8_t kaug[BWD_NST][4096];
  __align__(128) uint8_t qaug[2][256];
  alignas(16) float rowc[2][2][128];   // per item slot: -lse log2(e) and -D of its 128 query rows
  uint64_t qfull, qfree, full[BWD_NST], empty[BWD_NST], sfull, sfree, dpfull, dpfree, fin, finb;
  // per dS buffer: dS written (dsready) and the dQ product that read it done
  // (dqdone); a pair per buffer keeps each barrier within one phase of its
  // waiter (the elementwise warps may run a block ahead of thread B)
  uint64_t dsready[2], dqdone[2];
  uint64_t done[2];                       // per item slot: the item's dQ is complete
  uint64_t item_ready[2], item_free[2];   // per item slot: written by the producer / done with by the rest
  uint32_t tmem_base;
  int abort;
  // Two item slots, filled by the producer in turn: the item (-1 = no more), the
  // number of kv blocks its q block sees and their list, in order, with flags.
  int item[2], nlist[2];
  uint16_t list[2][BWD_MAXB];
  uint8_t lflags[2][BWD_MAXB];
};
static_assert(sizeof(DqSmem) + 1024 <= 227 * 1024, "dQ shared memory (+ 1 KB alignment slack)");

template <bool BF16, int MOD, bool DM>
__global__ void __launch_bounds__(BWD_T, 1) bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  DqSmem& sm = *reinterpret_cast<DqSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int BH = p.B * p.H;
  // Work items are (q block, b, h), numbered longest causal rows first.  CTAs
  // take them from the counter p.items in turn (one CTA per SM), or, with no
  // counter, one item each.
  const int n_items = p.nqb * BH;
  const bool persistent = p.items != nullptr;
  struct Item {
    int qb, bh, b, h;
  };
  auto item_of = [&](int L) {
    Item it;
    it.qb = p.nqb - 1 - L / BH;
    it.bh = L % BH;
    it.b = it.bh / p.H;
    it.h = it.bh % p.H;
    return it;
  };

  if (tid == 0) {
    mbar_init(smem_u32(&sm.qfull), 1);
    mbar_init(smem_u32(&sm.qfree), 1);   // thread A's commit after an item's score products
    for (int s = 0; s < BWD_NST; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 1);
    }
    mbar_init(smem_u32(&sm.sfull), 1);
    mbar_init(smem_u32(&sm.sfree), 256);
    mbar_init(smem_u32(&sm.dpfull), 1);
    mbar_init(smem_u32(&sm.dpfree), 256);
    mbar_init(smem_u32(&sm.dsready[0]), 256);
    mbar_init(smem_u32(&sm.dsready[1]), 256);
    mbar_init(smem_u32(&sm.dqdone[0]), 1);
    mbar_init(smem_u32(&sm.dqdone[1]), 1);
    mbar_init(smem_u32(&sm.fin), 1);
    mbar_init(smem_u32(&sm.finb), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&sm.done[t]), 1);
      mbar_init(smem_u32(&sm.item_ready[t]), 1);
      mbar_init(smem_u32(&sm.item_free[t]), 2 + 256);   // both MMA threads and every elementwise thread
    }
    sm.abort = 0;
    fence_mbar_init();
    fence_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  // The key-padding mask and (with `fold`) the ALiBi / checkerboard bias ride on
  // the S product, with the operands of the forward (fwd_d64.cu): checkerboard
  // (-1)^q t_i x (-1)^c (t = 0.5 / scale), ALiBi t_i x c / 128 (t = 128 slope_h /
  // scale, written into the item slot's query side by the producer), in three
  // 16-bit terms; ALiBi's slope_h (kv0 - q) is a per-row constant of each block.
  constexpr bool kModTerm = (MOD == MOD_ALIBI || MOD == MOD_CHECKER);
  const bool fold = kModTerm && p.fold;
  const bool aug = fold || p.km_bits != nullptr;
  if (aug) {
    uint4* z = reinterpret_cast<uint4*>(sm.kaug);
    for (int i = tid; i < (int)((BWD_NST * 4096 + 2 * 256) / 16); i += BWD_T) z[i] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    const uint16_t one = to16<BF16>(1.f);
    if (tid < 128 && fold) {
      const int r = tid;   // key column of a kv block
      uint16_t kt3[3];
      for (int i = 0; i < 3; ++i)
        kt3[i] = MOD == MOD_CHECKER ? ((r & 1) ? to16<BF16>(-1.f) : one) : to16<BF16>(float(r) * (1.f / 128.f));
      for (int st = 0; st < BWD_NST; ++st)
        for (int i = 0; i < 3; ++i) *reinterpret_cast<uint16_t*>(sm.kaug[st] + k16_offset(r, AUG_MOD + i)) = kt3[i];
    }
    if (tid >= 128 && tid < 128 + 16) {   // both slots' query sides: 8 rows each
      const int sl = (tid - 128) >> 3, r = tid & 7;
      uint8_t* o = sm.qaug[sl];
      *reinterpret_cast<uint16_t*>(o + k16_offset(r, AUG_KEY)) = one;
      if (MOD == MOD_CHECKER && fold) {
        uint16_t t[3];
        split3_plain<BF16>(0.5f * p.inv_scale, t);
        for (int i = 0; i < 3; ++i)   // a q block starts at a multiple of 128: the row's parity is r's
          *reinterpret_cast<uint16_t*>(o + k16_offset(r, AUG_MOD + i)) = (r & 1) ? uint16_t(t[i] ^ 0x8000u) : t[i];
      }
    }
    fence_async_smem();   // generic-proxy writes, read by the tensor core
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  // TMEM columns: S 128, dP 128, dS (16-bit pairs) 64 per buffer (blocks
  // alternate between two, so dS(u) is written while dQ += dS(u-1) K still
  // reads the other), dQ 64 per item slot
  constexpr uint32_t C_S = 0, C_DP = 128, C_DQ = 320;
  auto c_ds = [](uint32_t u) -> uint32_t { return (u & 1u) ? 448u : 256u; };

  if (warp == 0) {
    // ---- producer: takes the items and fills their slots (list of kv blocks, the
    // rows' -lse log2(e) and -D, the head's query-side term), loads an item's Q
    // and dO once the previous item's score products are done with them, then
    // streams its K / V blocks through the ring (continuing across items).
    WaitCtx c{&sm.abort, p.status, p.timeout_ns, 21};
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    int last_u[BWD_NST];
    for (int s = 0; s < BWD_NST; ++s) last_u[s] = -1;
    int u = 0, last_q = -1;
    bool ok = true;
    for (int ci = 0; ok; ++ci) {
      const int sl = ci & 1;
      int L = 0;
      if (lane == 0) L = persistent ? (int)atomicAdd(p.items, 1u) : (ci == 0 ? (int)blockIdx.x : n_items);
      L = __shfl_sync(0xffffffffu, L, 0);
      // the slot's previous item (ci - 2) is done with everywhere
      if (ci >= 2 && !wait_warp(smem_u32(&sm.item_free[sl]), ((ci - 2) >> 1) & 1, c)) break;
      if (L >= n_items) {   // no more items: the others stop at this slot
        if (lane == 0) {
          sm.item[sl] = -1;
          mbar_arrive(smem_u32(&sm.item_ready[sl]));
        }
        break;
      }
      const Item it = item_of(L);
      // the kv blocks this q block sees, in ascending order, 32 candidates per ballot
      int n = 0;
      for (int k0 = 0; k0 < p.nkb; k0 += 32) {
        const int kb = k0 + lane;
        bool keep = false;
        uint8_t fl = 0;
        if (kb < p.nkb) {
          const int ks = p.km_sum ? p.km_sum[it.b * p.nkb + kb] : 2;
          const int st =
              p.bm_tiles ? p.bm_tiles[it.b * p.bm_sb + it.h * p.bm_sh + (long long)it.qb * p.nkb + kb] : TILE_FULL;
          int ds = TILE_FULL;   // the dense tile state: dense build only
          if constexpr (DM)
            ds = p.dm.tiles[(((long long)it.b * p.dm.mb + (long long)it.h * p.dm.mh) * p.nqb + it.qb) * p.nkb + kb];
          keep = ks != 0 && st != TILE_EMPTY && ds != TILE_EMPTY;
          fl = (st == TILE_PARTIAL && p.bm_mod != MASKMOD_NONE ? KB_MASKMOD : 0) | (ks == 1 ? KB_KEYMASK : 0) |
               (ds == TILE_PARTIAL ? KB_DENSE : 0);
        }
        const unsigned m = __ballot_sync(0xffffffffu, keep);
        if (keep) {
          const int pos = n + __popc(m & ((1u << lane) - 1u));
          sm.list[sl][pos] = (uint16_t)kb;
          sm.lflags[sl][pos] = fl;
        }
        n += __popc(m);
      }
      {   // the rows' -lse log2(e) and -D (lane: rows 4 lane .. 4 lane + 3); rows past
          // Sq (partial last q block) get P = 0 and are not written
        const long long row = (long long)it.bh * p.Sq + it.qb * 128;
        float4 nl, nd;
        if ((p.Sq & 3) == 0 && it.qb * 128 + 128 <= p.Sq) {   // whole block, 16-byte aligned rows
          nl = __ldg(reinterpret_cast<const float4*>(p.lse2 + row) + lane);
          nd = __ldg(reinterpret_cast<const float4*>(p.delta + row) + lane);
        } else {
          float a[4], d[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const bool in = it.qb * 128 + 4 * lane + i < p.Sq;
            a[i] = in ? __ldg(p.lse2 + row + 4 * lane + i) : -INFINITY;
            d[i] = in ? __ldg(p.delta + row + 4 * lane + i) : 0.f;
          }
          nl = make_float4(a[0], a[1], a[2], a[3]);
          nd = make_float4(d[0], d[1], d[2], d[3]);
        }
        reinterpret_cast<float4*>(sm.rowc[sl][0])[lane] = nl;
        reinterpret_cast<float4*>(sm.rowc[sl][1])[lane] = nd;
      }
      if (lane == 0) {
        sm.item[sl] = L;
        sm.nlist[sl] = n;
        if (MOD == MOD_ALIBI && fold) {
          // the head's factor of the folded slope_h c term in the slot's query side
          // (one thread at fixed offsets: stores from every lane of the producer
          // cost the kernel registers)
          uint16_t t3[3];
          split3_plain<BF16>(128.f * exp2f(-8.0f * float(it.h + 1) / float(p.H)) * p.inv_scale, t3);
#pragma unroll
          for (int r = 0; r < 8; ++r)
            for (int e = 0; e < 3; ++e)
              *reinterpret_cast<uint16_t*>(sm.qaug[sl] + k16_offset(r, AUG_MOD + e)) = t3[e];
          fence_async_smem();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.item_ready[sl]));   // release: the slot is visible to its waiters
      // Q and dO of the item, once the previous item's score products are done with them
      if (ci >= 1 && !wait_warp(smem_u32(&sm.qfree), (ci - 1) & 1, c)) break;
      if (lane == 0) {
        mbar_expect_tx(smem_u32(&sm.qfull), 2 * BWD_TILE);
        tma_load_2d(smem_u32(sm.q), &p.tm_q, smem_u32(&sm.qfull), 0, it.bh * p.Sq + it.qb * 128);
        tma_load_2d(smem_u32(sm.dO), &p.tm_do, smem_u32(&sm.qfull), 0, it.bh * p.Sq + it.qb * 128);
      }
      last_q = ci;
      for (int j = 0; j < n; ++j) {
        const int s = u % BWD_NST;
        if (u >= BWD_NST && !wait_warp(smem_u32(&sm.empty[s]), ((u / BWD_NST) - 1) & 1, c)) {
          ok = false;
          break;
        }
        const int kb = sm.list[sl][j];
        if (aug && p.km_bits) {   // lane owns keys 4 lane .. 4 lane + 3: column AUG_KEY of kaug[s]
          uint32_t bits = 0xffffffffu;
          if (sm.lflags[sl][j] & KB_KEYMASK) bits = km_word(p.km_bits, it.b, p.Skv, kb * 128 + 4 * lane);
          // the infinity whose product with the scale is -inf (scale != 0)
          const uint16_t ninf = p.sc < 0.f ? (BF16 ? 0x7F80u : 0x7C00u) : (BF16 ? 0xFF80u : 0xFC00u);
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = 4 * lane + i;
            *reinterpret_cast<uint16_t*>(sm.kaug[s] + k16_offset(col, AUG_KEY)) =
                ((bits >> (col & 31)) & 1u) ? uint16_t(0) : ninf;
          }
          fence_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          const uint32_t fb = smem_u32(&sm.full[s]);
          mbar_expect_tx(fb, 2 * BWD_TILE);   // release: the bias column above is visible to its waiters
          tma_load_2d(smem_u32(sm.k[s]), &p.tm_k, fb, 0, it.bh * p.Skv + kb * 128);
          tma_load_2d(smem_u32(sm.v[s]), &p.tm_v, fb, 0, it.bh * p.Skv + kb * 128);
        }
        last_u[s] = u;
        ++u;
      }
    }
    if (lane == 0) {   // every copy issued has landed before the CTA exits (instant unless aborted)
      if (last_q >= 0) drain_wait(smem_u32(&sm.qfull), last_q & 1, p.timeout_ns);
      for (int s = 0; s < BWD_NST; ++s)
        if (last_u[s] >= 0) drain_wait(smem_u32(&sm.full[s]), (last_u[s] / BWD_NST) & 1, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issue, thread A: S = Q K^T (+ column terms) and dP = dO V^T, each
    // issued as soon as the elementwise warps hold the previous one in registers
    // (u counts blocks over all items of the CTA: the barriers' phases).
    if (lane == 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 22};
      constexpr uint32_t ID_SS = idesc_f16(128, 128, BF16, false, false);
      const uint64_t qd = sdesc_sw128(smem_u32(sm.q), 16, 1024), od = sdesc_sw128(smem_u32(sm.dO), 16, 1024);
      uint32_t u = 0;
      bool ok = true;
      for (int ci = 0; ok; ++ci) {
        const int sl = ci & 1;
        if (!wait_one(smem_u32(&sm.item_ready[sl]), (ci >> 1) & 1, c)) break;
        if (sm.item[sl] < 0) break;
        const int n = sm.nlist[sl];
        const uint64_t qad = sdesc_k16_rows8(smem_u32(sm.qaug[sl]));
        if (!wait_one(smem_u32(&sm.qfull), ci & 1, c)) break;
        for (int j = 0; j < n; ++j, ++u) {
          const int s = u % BWD_NST;
          if (!wait_one(smem_u32(&sm.full[s]), (u / BWD_NST) & 1, c)) { ok = false; break; }
          if (u > 0 && !wait_one(smem_u32(&sm.sfree), (u - 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
          {   // S_u = Q K_u^T (+ column terms)
            const uint64_t kd = sdesc_sw128(smem_u32(sm.k[s]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + C_S, qd + 2 * kk, kd + 2 * kk, ID_SS, kk > 0);
            if (aug) mma_ss(tmem + C_S, qad, sdesc_k16(smem_u32(sm.kaug[s])), ID_SS, 1u);
            tc_commit(smem_u32(&sm.sfull));
          }
          if (u > 0 && !wait_one(smem_u32(&sm.dpfree), (u - 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
          {   // dP_u = dO V_u^T
            const uint64_t vd = sdesc_sw128(smem_u32(sm.v[s]), 16, 1024);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) mma_ss(tmem + C_DP, od + 2 * kk, vd + 2 * kk, ID_SS, kk > 0);
            tc_commit(smem_u32(&sm.dpfull));
          }
        }
        if (!ok) break;
        // both arrive once this item's score products are complete: Q and dO may be
        // reloaded, and the slot (its query side) refilled
        tc_commit(smem_u32(&sm.qfree));
        tc_commit(smem_u32(&sm.item_free[sl]));
      }
      // every MMA issued by this thread completes before the CTA lets go of TMEM
      tc_commit(smem_u32(&sm.fin));
      drain_wait(smem_u32(&sm.fin), 0, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 10) {
    // ---- MMA issue, thread B: dQ += dS K, A operand from TMEM where the
    // elementwise warps left dS; the dQ accumulator alternates between two TMEM
    // regions by item slot, so an item's products need not wait for the previous
    // item's epilogue (a slot is refilled only after its epilogue).
    if (lane == 0) {
      WaitCtx c{&sm.abort, p.status, p.timeout_ns, 24};
      constexpr uint32_t ID_TS = idesc_f16(128, 64, BF16, false, true);
      uint32_t u = 0;
      bool ok = true;
      for (int ci = 0; ok; ++ci) {
        const int sl = ci & 1;
        if (!wait_one(smem_u32(&sm.item_ready[sl]), (ci >> 1) & 1, c)) break;
        if (sm.item[sl] < 0) break;
        const int n = sm.nlist[sl];
        const uint32_t tdq = tmem + C_DQ + 64 * sl;
        for (int j = 0; j < n; ++j, ++u) {
          const int s = u % BWD_NST;
          if (!wait_one(smem_u32(&sm.full[s]), (u / BWD_NST) & 1, c)) { ok = false; break; }
          if (!wait_one(smem_u32(&sm.dsready[u & 1]), (u >> 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
          const uint64_t kd = sdesc_sw128(smem_u32(sm.k[s]), 8192, 1024);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            mma_ts(tdq, tmem + c_ds(u) + 8 * kk, kd + 128 * kk, ID_TS, (j > 0 || kk > 0));
          tc_commit(smem_u32(&sm.dqdone[u & 1]));
          tc_commit(smem_u32(&sm.empty[s]));
        }
        if (!ok) break;
        tc_commit(smem_u32(&sm.done[sl]));   // this item's dQ is complete once it arrives
        mbar_arrive(smem_u32(&sm.item_free[sl]));
      }
      tc_commit(smem_u32(&sm.finb));
      drain_wait(smem_u32(&sm.finb), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    const int w = (warp - 2) >> 2;   // kv columns [64 w, 64 w + 64)
    const int quad = warp & 3;
    const int r = 32 * quad + lane;
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    WaitCtx c{&sm.abort, p.status, p.timeout_ns, 23 + w};
    const uint64_t scv = f2(p.sc, p.sc);
    uint32_t u = 0;   // blocks over all items (the barriers' phases)
    bool ok = true;
    for (int ci = 0; ok; ++ci) {
      const int sl = ci & 1;
      if (!wait_warp(smem_u32(&sm.item_ready[sl]), (ci >> 1) & 1, c)) break;
      const int L = sm.item[sl];
      if (L < 0) break;
      const Item it = item_of(L);
      const int qb = it.qb, bh = it.bh, b = it.b, h = it.h;
      const int N = sm.nlist[sl];
      const int q = qb * 128 + r;
      const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
      const float nl2 = sm.rowc[sl][0][r];   // -lse log2(e); -inf past Sq
      const float nd = sm.rowc[sl][1][r];    // -D
      const uint64_t nl2v = f2(nl2, nl2), ndv = f2(nd, nd);
      for (int j = 0; j < N; ++j, ++u) {
        const int kb = sm.list[sl][j];
        const uint8_t f = sm.lflags[sl][j];
        const int k0 = kb * 128 + 64 * w;   // first key of this half
        const bool causal = (MOD == MOD_CAUSAL && kb * 128 + 127 > qb * 128) ||
                            ((f & KB_MASKMOD) && p.bm_mod == MASKMOD_CAUSAL);
        const bool umask = MOD == MOD_USER && (f & KB_MASKMOD) && p.bm_mod == MASKMOD_USER;
        // keep column cc of this half iff cc <= lim: the causal limit and, in a
        // partial last kv block, the end of the keys
        const int kvl = p.Skv - 1 - k0;
        const bool limited = causal || kvl < 63;
        const int lim = causal ? min(q - k0, kvl) : kvl;
        // this row's dense-mask bits for the half's 64 keys
        bool dense = false;
        uint2 dwv = make_uint2(0u, 0u);
        if constexpr (DM) {
          dense = f & KB_DENSE;
          const long long dmi = (long long)b * p.dm.mb + (long long)h * p.dm.mh;
          if (dense && q < p.Sq)
            dwv = __ldg(reinterpret_cast<const uint2*>(p.dm.rowbits + (dmi * p.Sq + q) * (4LL * p.nkb) + 4 * kb +
                                                       2 * w));
        }
        // the block's bias constants, ahead of the wait (they do not depend on S)
        uint64_t chk = 0;
        if constexpr (MOD == MOD_CHECKER) {
          const float hb = ((q + k0) & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;   // even column
          chk = f2(hb, -hb);
        }
        const float abase = (MOD == MOD_ALIBI) ? slope2 * float(k0 - q) : 0.f;
        // with the bias folded into S, all that is left per pair is this row's constant
        const float fb = (MOD == MOD_ALIBI) ? slope2 * float(kb * 128 - q) : 0.f;
        const uint64_t addf = fadd2(nl2v, f2(fb, fb));
        if (!wait_warp(smem_u32(&sm.sfull), u & 1, c)) { ok = false; break; }
        tc_fence_after();
        uint32_t rr[64];
        tmem_ld64(tmem + lane_off + C_S + 64 * w, rr);
        // S(u) is in registers: the next S may be computed over it
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.sfree));
        float pr[64];
        // one straight-line copy per causal/not: no runtime test inside the unrolled loop
        auto probs = [&](auto causal_c, auto dense_c, auto fold_c) {
          constexpr bool CAUSAL = decltype(causal_c)::value;
          constexpr bool DENSE = decltype(dense_c)::value;
          constexpr bool FOLD = decltype(fold_c)::value;
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            uint64_t add = FOLD ? addf : nl2v;
            if constexpr (MOD == MOD_CHECKER && !FOLD) add = fadd2(add, chk);
            if constexpr (MOD == MOD_ALIBI && !FOLD)
              add = fadd2(add, f2(fmaf(slope2, float(2 * i), abase), fmaf(slope2, float(2 * i + 1), abase)));
            float x0, x1;
            unf2(ffma2(f2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1])), scv, add), x0, x1);
            if constexpr (MOD == MOD_USER) {
              x0 = fmaf(user_bias(b, h, q, k0 + 2 * i), kLog2e, x0);
              x1 = fmaf(user_bias(b, h, q, k0 + 2 * i + 1), kLog2e, x1);
              if (umask) {   // a PARTIAL tile of a user mask_mod's block mask
                x0 = user_keep(b, h, q, k0 + 2 * i) ? x0 : -INFINITY;
                x1 = user_keep(b, h, q, k0 + 2 * i + 1) ? x1 : -INFINITY;
              }
            }
            if (CAUSAL) {
              x0 = 2 * i > lim ? -INFINITY : x0;
              x1 = 2 * i + 1 > lim ? -INFINITY : x1;
            }
            if constexpr (DENSE) {
              const uint32_t dwi = i < 16 ? dwv.x : dwv.y;
              x0 = (dwi & (1u << ((2 * i) & 31))) ? x0 : -INFINITY;
              x1 = (dwi & (1u << ((2 * i + 1) & 31))) ? x1 : -INFINITY;
            }
            pr[2 * i] = ex2(x0);
            pr[2 * i + 1] = ex2(x1);
          }
        };
        auto probs_any = [&](auto fold_c) {
          if (dense) {   // with dense bits, the limited copy too (never with DM = false)
            if constexpr (DM) probs(bconst<true>{}, bconst<true>{}, fold_c);
          } else if (limited) {
            probs(bconst<true>{}, bconst<false>{}, fold_c);
          } else {
            probs(bconst<false>{}, bconst<false>{}, fold_c);
          }
        };
        if constexpr (kModTerm) {
          if (fold) probs_any(bconst<true>{});
          else probs_any(bconst<false>{});
        } else {
          probs_any(bconst<false>{});
        }
        if (!wait_warp(smem_u32(&sm.dpfull), u & 1, c)) { ok = false; break; }
        tc_fence_after();
        tmem_ld64(tmem + lane_off + C_DP + 64 * w, rr);
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.dpfree));
        uint32_t dsk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          float d0, d1;
          unf2(fmul2(f2(pr[2 * i], pr[2 * i + 1]),
                     fadd2(f2(__uint_as_float(rr[2 * i]), __uint_as_float(rr[2 * i + 1])), ndv)),
               d0, d1);
          dsk[i] = pack2<BF16>(d0, d1);
        }
        // dQ(u-2) has finished reading this dS buffer (dqdone[b] completes once per
        // use of buffer b = u & 1: the use before this one is phase (u - 2) / 2)
        if (u > 1) {
          if (!wait_warp(smem_u32(&sm.dqdone[u & 1]), ((u - 2) >> 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st32(tmem + lane_off + c_ds(u) + 32 * w, dsk);
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.dsready[u & 1]));
      }
      tmem_st_wait();
      if (!ok) break;
      if (w == 0) {   // epilogue: warps 2-5 write the dQ rows (scaled)
        if (!wait_warp(smem_u32(&sm.done[sl]), (ci >> 1) & 1, c)) break;
        tc_fence_after();
        uint32_t rr[64], o[32];
        if (N > 0) {
          tmem_ld64(tmem + lane_off + C_DQ + 64 * sl, rr);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) rr[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          o[i] = pack2<BF16>(__uint_as_float(rr[2 * i]) * p.scale, __uint_as_float(rr[2 * i + 1]) * p.scale);
        uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.dq) + ((size_t)bh * p.Sq + q) * 64);
        if (q < p.Sq) {
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        }
      }
      // this item's slot (and, once its epilogue has read it, its dQ region) is done with
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.item_free[sl]));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, 512);
  // the last CTA to finish re-arms the item counter for the next call (this
  // thread made the CTA's last claim, so every claim precedes the reset)
  if (persistent && tid == 0) {
    __threadfence();
    if (atomicAdd(p.items + 1, 1u) == gridDim.x - 1u) {
      p.items[0] = 0u;
      p.items[1] = 0u;
    }
  }
  // Launched with programmatic dependent launch behind the dK/dV pass, whose
  // results it does not read (the preprocess it needs was complete before that
  // pass let it launch): it waits for that grid only here, so that its own
  // completion still implies the whole backward's for later work in the stream.
  if (tid == 0) griddep_wait();
}

// ---------------------------------------------------------------------------
#ifndef __CUDACC_RTC__
// Both passes are launched with programmatic dependent launch (the dK/dV pass
// behind the preprocess, the dQ pass behind the dK/dV pass); see the kernels.
static cudaError_t launch_bwd_pdl(const BwdParams& p, const void* kern, bool dkdv, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.items ? p.ctas : p.B * p.H * (dkdv ? p.nkb : p.nqb)));
  cfg.blockDim = dim3(BWD_T);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  void* args[] = {const_cast<BwdParams*>(&p)};
  return cudaLaunchKernelExC(&cfg, kern, args);
}

// Backward kernels of these layouts built elsewhere (a run-time-compiled
// score_mod): the same shared memory, grid and block as the built-in variants.
cudaError_t launch_bwd_kernel(const BwdParams& p, const void* kern, bool dkdv, cudaStream_t st) {
  const size_t smem = (dkdv ? sizeof(DkdvSmem) : sizeof(DqSmem)) + 1024;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  return launch_bwd_pdl(p, kern, dkdv, smem, st);
}

template <typename Smem, bool BF16, int MOD, bool DKDV>
static cudaError_t launch_bwd_t(const BwdParams& p, cudaStream_t st) {
  // DM: the build with the dense-mask path, used only when a dense mask is given
  auto plain = DKDV ? bwd_dkdv_kernel<BF16, MOD, false> : bwd_dq_kernel<BF16, MOD, false>;
  auto masked = DKDV ? bwd_dkdv_kernel<BF16, MOD, true> : bwd_dq_kernel<BF16, MOD, true>;
  auto kern = p.dm.tiles ? masked : plain;
  const size_t smem = sizeof(Smem) + 1024;
  static const cudaError_t e0 = cudaFuncSetAttribute(plain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  static const cudaError_t e1 = cudaFuncSetAttribute(masked, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  const cudaError_t e = p.dm.tiles ? e1 : e0;
  if (e != cudaSuccess) return e;
  return launch_bwd_pdl(p, reinterpret_cast<const void*>(kern), DKDV, smem, st);
}

template <typename Smem, bool DKDV>
static cudaError_t launch_bwd_any(const BwdParams& p, bool bf16, int mod, cudaStream_t st) {
  if (bf16) {
    switch (mod) {
      case MOD_NONE: return launch_bwd_t<Smem, true, MOD_NONE, DKDV>(p, st);
      case MOD_ALIBI: return launch_bwd_t<Smem, true, MOD_ALIBI, DKDV>(p, st);
      case MOD_CHECKER: return launch_bwd_t<Smem, true, MOD_CHECKER, DKDV>(p, st);
      default: return launch_bwd_t<Smem, true, MOD_CAUSAL, DKDV>(p, st);
    }
  }
  switch (mod) {
    case MOD_NONE: return launch_bwd_t<Smem, false, MOD_NONE, DKDV>(p, st);
    case MOD_ALIBI: return launch_bwd_t<Smem, false, MOD_ALIBI, DKDV>(p, st);
    case MOD_CHECKER: return launch_bwd_t<Smem, false, MOD_CHECKER, DKDV>(p, st);
    default: return launch_bwd_t<Smem, false, MOD_CAUSAL, DKDV>(p, st);
  }
}

cudaError_t launch_bwd_dkdv(const BwdParams& p, bool bf16, int mod, cudaStream_t st) {
  return launch_bwd_any<DkdvSmem, true>(p, bf16, mod, st);
}
cudaError_t launch_bwd_dq(const BwdParams& p, bool bf16, int mod, cudaStream_t st) {
  return launch_bwd_any<DqSmem, false>(p, bf16, mod, st);
}

#endif  // host

}  // namespace attn
