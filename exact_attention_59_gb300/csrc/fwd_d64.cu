// fwd_d64.cu - prefill forward, head dim 64, f16/bf16, tcgen05 + TMA.
//
// The online-softmax forward of the attnax Pallas kernel body (per kv block:
// scores = q k^T scale, score_mod, mask, m_new = max(m, rowmax),
// alpha = exp(m - m_new), p = exp(s - m_new), l = l alpha + sum p,
// acc = acc alpha + p v; finally o = acc / l), in base 2 as the flaxattention
// README's "log2 trick": the scale and the mods' biases carry a log2(e) factor
// and every exp is one MUFU ex2.
//
// A work item is two 128-row query tiles of one (b, h); the CTA streams the
// union of their kv-block lists once.  The grid is one CTA per SM (at most one
// per item), and the CTAs take items from an atomic counter in the workspace,
// longest causal pairs first (the pairs past the last full round may be
// claimed as single query tiles, so that the partly filled last round runs on
// more CTAs); the split variant (a chunk of queries, or a kv range per CTA)
// runs one item per CTA instead.  Items pass through two slots
// (the item and its kv-block flags), so the next item's query tiles and first
// blocks load while the softmax finishes the previous one.
//   warp 0      producer: takes the items, fills the slots, loads both Q tiles of
//               an item into its slot's buffers (two items' query tiles are
//               resident, so an item's tiles load while the previous item runs),
//               then K and V tiles of each kv block into a FWD_NST-stage ring
//               (128B swizzle, 16 KB per tile), continuing across items.
//   warps 1-2   warp 1 allocates 512 TMEM columns; lane 0 of warp 1 + t issues
//               tile t's tcgen05.mma: S_t = Q_t K^T (128x128, f32 in TMEM) and
//               O_t += P_t V with P_t read from TMEM.  One issuing thread per
//               tile, so that a wait for one tile's P or free S never holds
//               back the other tile's products (one thread issuing both tiles'
//               products in a fixed order was ~30% slower), and S_t(n+1) is
//               issued as soon as the softmax has copied S_t(n) to registers,
//               so it overlaps the exponentials.
//   warps 3-6   softmax of tile 0, warps 7-10 softmax of tile 1: one thread per
//               query row (TMEM lane), 128 scores per kv block in registers,
//               running max/sum per thread, P packed to 16-bit into TMEM,
//               O rescaled in TMEM when the row max grows, then the epilogue.
// TMEM columns per tile t: S [256t, 256t+128), P [256t+128, 256t+192),
// O [256t+192, 256t+256).
#include "kernels.h"

namespace attn {

struct __align__(1024) FwdSmem {
  uint8_t q[2][2][FWD_TILE_BYTES];   // per item slot: the item's two query tiles
  uint8_t k[FWD_NST][FWD_TILE_BYTES];
  uint8_t v[FWD_NST][FWD_TILE_BYTES];
  // Column terms folded into S = Q K^T as one more K = 16 step (K = 16 operands
  // without swizzle, 4 KB each; columns as AUG_MOD / AUG_KEY in common.cuh):
  // qaug (per query row, resident) x kaug[s] (per key of stage s).
  __align__(128) uint8_t qaug[4096];
  __align__(128) uint8_t kaug[FWD_NST][4096];
  __align__(128) uint8_t qaug_h[2][256];   // folded ALiBi: an item slot's query side (8 rows, repeated)
  uint64_t full[FWD_NST], empty[FWD_NST];
  uint64_t qfull[2], sfull[2], sfree[2], pready[2], odone[2], fin[2];   // qfull: per item slot
  uint64_t item_ready[2], item_free[2];   // per item slot: written by the producer / done with by the rest
  alignas(16) float cb[FWD_NST][2][128];   // per-stage column bias (log2 units): key mask, ALiBi column term, checkerboard
  uint32_t tmem_base;
  int abort;
  // Two item slots, filled by the producer in turn: the item (-1 = no more) and
  // its flags per tile and kv block.
  int item[2];
  uint8_t flags[2][2][FWD_MAXKB];
};

// the bias table is read 16 bytes at a time
#ifndef __CUDACC_RTC__   // (the offline build checks the same layout)
static_assert(offsetof(FwdSmem, cb) % 16 == 0, "cb must be 16-byte aligned");
#endif

// Pass 1 over one row's 128 scores of a kv block: x = s * scale (+ column bias
// from the stage's table), -inf for columns cc > lim (the causal rule, or keys
// past the end in a partial last block) and, with DENSE, for columns whose bit
// in the row's dense-mask words dw is 0; and the running maximum in four
// independent chains.
// With USER, x += user_bias(b, h, q, kv0 + cc) log2(e) (a run-time-compiled score_mod)
// and, with UMASK (a PARTIAL tile of a user mask_mod's block mask), -inf where
// user_keep(b, h, q, kv0 + cc) is false.
// With RAW (no table, no user bias, scale > 0) the scores stay unscaled: the
// masks and the maximum work on s itself (max of s * scale = scale * max of s),
// and the exponential pass applies the scale in its one FFMA.
// N = the columns passed: column cc here is column cc of the caller's share,
// whose table `tb`, limit `lim`, dense words `dw` (x = its columns 0-31,
// y = 32-63, ...) and first key `ukv0` the caller has offset to that share.
template <int N, bool TABLE, bool LIMITED, bool DENSE, bool USER = false, bool RAW = false, bool UMASK = false>
DEVI void scale_scores(uint32_t (&r)[N], uint64_t scv, const float* tb, int lim, uint4 dw, float (&mx)[4],
                       int ub = 0, int uh = 0, int uq = 0, int ukv0 = 0) {
#pragma unroll
  for (int i = 0; i < N / 2; i += 2) {
    float4 bias = make_float4(0.f, 0.f, 0.f, 0.f);
    if (TABLE) bias = *reinterpret_cast<const float4*>(tb + 2 * i);
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int c = 2 * (i + j);
      const uint64_t sv = f2(__uint_as_float(r[c]), __uint_as_float(r[c + 1]));
      const uint64_t xv = TABLE ? ffma2(sv, scv, j ? f2(bias.z, bias.w) : f2(bias.x, bias.y))
                                : (RAW ? sv : fmul2(sv, scv));
      float x0, x1;
      unf2(xv, x0, x1);
      if constexpr (USER) {
        x0 = fmaf(user_bias(ub, uh, uq, ukv0 + c), kLog2e, x0);
        x1 = fmaf(user_bias(ub, uh, uq, ukv0 + c + 1), kLog2e, x1);
      }
      if constexpr (UMASK) {
        x0 = user_keep(ub, uh, uq, ukv0 + c) ? x0 : -INFINITY;
        x1 = user_keep(ub, uh, uq, ukv0 + c + 1) ? x1 : -INFINITY;
      }
      if (LIMITED) {
        x0 = c > lim ? -INFINITY : x0;
        x1 = c + 1 > lim ? -INFINITY : x1;
      }
      if constexpr (DENSE) {
        const uint32_t w = c < 32 ? dw.x : (c < 64 ? dw.y : (c < 96 ? dw.z : dw.w));
        x0 = (w & (1u << (c & 31))) ? x0 : -INFINITY;
        x1 = (w & (1u << ((c + 1) & 31))) ? x1 : -INFINITY;
      }
      r[c] = __float_as_uint(x0);
      r[c + 1] = __float_as_uint(x1);
      mx[(i + j) & 3] = fmax3(mx[(i + j) & 3], x0, x1);
    }
  }
}

// Kernel variants, so that each path costs the others nothing:
//   FWD_PLAIN  the forward;
//   FWD_DENSE  with the dense-mask path;
//   FWD_CHUNK  queries at a position offset, kv blocks split over CTAs (decode).
constexpr int FWD_PLAIN = 0, FWD_DENSE = 1, FWD_CHUNK = 2;


// Keys key .. key + 3 of batch row b of a byte key mask (nonzero = keep; keys
// at or past Skv count as masked), as the low 4 bits.
DEVI uint32_t key_bits4(const uint8_t* km, int b, int Skv, int key) {
  const uint8_t* row = km + (size_t)b * Skv;
  if (key + 4 <= Skv && ((reinterpret_cast<uintptr_t>(row + key) & 3) == 0)) {
    const uint32_t w = __ldg(reinterpret_cast<const uint32_t*>(row + key));
    return ((w & 0xffu) ? 1u : 0u) | ((w & 0xff00u) ? 2u : 0u) | ((w & 0xff0000u) ? 4u : 0u) |
           ((w & 0xff000000u) ? 8u : 0u);
  }
  uint32_t r = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i)
    if (key + i < Skv && __ldg(row + key + i) != 0) r |= 1u << i;
  return r;
}

// Key block kb of batch row b of a byte key mask: 0 no key kept, 1 some, 2 all
// (of the block's keys below Skv).  A whole, 16-byte aligned block is read as
// eight independent 16-byte loads and its nonzero bytes counted four at a time.
DEVI int key_block_summary(const uint8_t* km, int b, int Skv, int kb) {
  const int k0 = kb * 128, valid = min(128, Skv - k0);
  const uint8_t* row = km + (size_t)b * Skv + k0;
  int kept = 0;
  if (valid == 128 && (reinterpret_cast<uintptr_t>(row) & 15) == 0) {
    uint4 v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldg(reinterpret_cast<const uint4*>(row) + i);
#pragma unroll
    for (int i = 0; i < 8; ++i)
      kept += __popc(__vcmpne4(v[i].x, 0u)) + __popc(__vcmpne4(v[i].y, 0u)) + __popc(__vcmpne4(v[i].z, 0u)) +
              __popc(__vcmpne4(v[i].w, 0u));
    kept >>= 3;   // 8 bits per nonzero byte
  } else {
    for (int i = 0; i < valid; ++i) kept += __ldg(row + i) != 0 ? 1 : 0;
  }
  return kept == 0 ? 0 : (kept == valid ? 2 : 1);
}

// A lane's key-mask word for keys key .. key + 3 (key a multiple of 4): bit
// (key + i) mod 32 is key + i's keep bit, from the packed bits or, without them,
// from the byte mask (the other bits are not used).
DEVI uint32_t lane_key_bits(const FwdParams& p, int b, int key) {
  if (p.km_bits) return km_word(p.km_bits, b, p.Skv, key);
  return key_bits4(p.km, b, p.Skv, key) << (key & 31);
}

template <bool BF16, int MOD, int VAR>
__global__ void __launch_bounds__(FWD_THREADS, 1) fwd_d64_kernel(const __grid_constant__ FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  FwdSmem& sm = *reinterpret_cast<FwdSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  constexpr bool DM = VAR == FWD_DENSE, CHUNK = VAR == FWD_CHUNK;
  // the waits' slow paths take their context by address in the run-time-compiled
  // score_mod build (measured faster there, and slower in the built-in mods)
  using WC = WaitCtxT<MOD == MOD_USER>;
  const int BH = p.B * p.H;
  const int n_items = p.npairs * BH;   // (pair of query tiles, b, h), longest causal pairs first
  // The split variant runs one item per CTA over its range of kv blocks.  Otherwise
  // CTAs take items from the counter p.items in turn (one CTA per SM), or, with no
  // counter, one item each, blockIdx.x.
  const int split = CHUNK ? blockIdx.x / n_items : 0;   // kv-block range of this CTA
  const int kb_lo = CHUNK ? split * p.kps : 0;
  const int kb_hi = CHUNK && p.nsplit > 1 ? min(p.nkb, kb_lo + p.kps) : p.nkb;
  const int q_off = CHUNK ? p.q_off : 0;
  const bool persistent = !CHUNK && p.items != nullptr;
  const bool singles = persistent && p.single_tail;
  const int n_claims = singles ? p.n_whole + 2 * (n_items - p.n_whole) : n_items;
  // an item's coordinates (a single-tile item keeps its tile in slot 0 and
  // leaves slot 1 empty, as the last pair of an odd tile count does)
  struct Item {
    int bh, b, h, qt0, qt1;
    bool valid1;
  };
  auto item_of = [&](int L) {
    Item it;
    int which = -1;   // single-tile item: the pair's tile 0 or 1
    if (singles && L >= p.n_whole) {
      which = (L - p.n_whole) & 1;
      L = p.n_whole + ((L - p.n_whole) >> 1);
    }
    const int pair = p.npairs - 1 - L / BH;
    it.bh = L % BH;
    it.b = it.bh / p.H;
    it.h = it.bh % p.H;
    it.qt0 = 2 * pair + (which == 1 ? 1 : 0);
    it.qt1 = which >= 0 ? p.nqb : 2 * pair + 1;
    it.valid1 = it.qt1 < p.nqb;
    return it;
  };
  if constexpr (CHUNK) {
    // launched with programmatic dependent launch: this CTA's first K and V rows
    // (kv blocks from kb_lo, contiguous, 128 bytes a row) go towards L2, the next
    // grid may launch, and nothing is read or written before the grids ahead of
    // this one have completed (L2 is the point of coherence: a line fetched
    // early still reflects writes made before the wait)
    const int bh0 = item_of(blockIdx.x % n_items).bh;
    if (tid < 2 && p.kraw && p.vraw) {   // (at most 2 FWD_NST blocks: the ring streams the rest)
      const long long r0 = (long long)bh0 * p.Skv + (long long)kb_lo * 128;
      const long long r1 = (long long)bh0 * p.Skv + min((long long)p.Skv, (long long)min(kb_hi, kb_lo + 2 * FWD_NST) * 128);
      if (r1 > r0)
        prefetch_l2_bulk(static_cast<const unsigned char*>(tid == 0 ? p.kraw : p.vraw) + r0 * 128,
                         static_cast<uint32_t>((r1 - r0) * 128));
    }
    griddep_launch_dependents();
    griddep_wait();
  } else {
    // a grid launched behind this one with programmatic dependent launch (the
    // backward preprocess) may start on SMs this grid leaves idle; it waits for
    // this grid before it reads anything this grid writes
    griddep_launch_dependents();
  }

  // ---- setup: barriers, TMEM (the items' flags and query tiles come from the producer)
  if (tid == 0) {
    for (int s = 0; s < FWD_NST; ++s) {
      mbar_init(smem_u32(&sm.full[s]), 1);
      mbar_init(smem_u32(&sm.empty[s]), 2);   // one arrival per tile per kv block (a tile with no rows arrives too)
    }
    mbar_init(smem_u32(&sm.qfull[0]), 1);
    mbar_init(smem_u32(&sm.qfull[1]), 1);
    for (int t = 0; t < 2; ++t) {
      mbar_init(smem_u32(&sm.sfull[t]), 1);
      mbar_init(smem_u32(&sm.sfree[t]), 128);
      mbar_init(smem_u32(&sm.pready[t]), 128);
      mbar_init(smem_u32(&sm.odone[t]), 1);
      mbar_init(smem_u32(&sm.fin[t]), 1);
      mbar_init(smem_u32(&sm.item_ready[t]), 1);
      mbar_init(smem_u32(&sm.item_free[t]), 2 + 256);   // both MMA threads and every softmax thread
    }
    sm.abort = 0;
    fence_mbar_init();
    fence_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(&sm.tmem_base), 512);
    tmem_relinquish();
  }
  constexpr bool kTableMod = (MOD == MOD_ALIBI || MOD == MOD_CHECKER);
  // Terms that depend on the query row or the key column alone ride on the S
  // product as one more K = 16 step (the tensor core adds them; the softmax warps
  // do no per-score work for them):
  //   key-padding mask: 1 x (0 or -inf) in column AUG_KEY (exact: +0 or -inf);
  //   with `fold`, the mod's bias over scale in columns AUG_MOD .. +2, as three
  //   16-bit terms of one f32 value:
  //     checkerboard  (-1)^q_pos t_i  x  (-1)^c        (t = 0.5 / scale)
  //     ALiBi         t_i             x  c / 128       (t = 128 slope_h / scale)
  //   c = key column in the block (a kv block starts at a multiple of 128, so
  //   (-1)^kv = (-1)^c; c / 128 is exact in both 16-bit types, and each product
  //   t_i c / 128 is exact in f32); ALiBi's t depends on the head: its query
  //   side is the same in every row, 8 rows per item slot (qaug_h) that the
  //   descriptor repeats over the tile, written by the producer with the
  //   slot's flags.  ALiBi's remaining
  //   slope_h (kv0 - q_pos) is a constant per row and block, added to the row
  //   maximum (below).  Without `fold` (scale 0,
  //   or a bias too large for three 16-bit terms) the producer's per-column table
  //   carries the mod and the mask instead.
  const bool fold = kTableMod && p.fold;
  const bool use_table = kTableMod && !fold;   // the table then carries the key mask too
  const bool kmask = p.km_bits != nullptr || p.km != nullptr;
  const bool aug = !use_table && (fold || kmask);
  if (aug) {
    uint4* z = reinterpret_cast<uint4*>(sm.qaug);
    for (int i = tid; i < (1 + FWD_NST) * 4096 / 16; i += FWD_THREADS) z[i] = make_uint4(0u, 0u, 0u, 0u);
    if (tid < 2 * 256 / 16) reinterpret_cast<uint4*>(sm.qaug_h)[tid] = make_uint4(0u, 0u, 0u, 0u);
    __syncthreads();
    if (tid < 128) {
      const int r = tid;   // query row of the tile, and key column of a block
      const uint16_t one = to16<BF16>(1.f);
      *reinterpret_cast<uint16_t*>(sm.qaug + k16_offset(r, AUG_KEY)) = one;
      if (fold) {
        uint16_t qt3[3], kt3[3];
        if constexpr (MOD == MOD_CHECKER) {
          uint16_t t[3];
          split3_plain<BF16>(0.5f * p.inv_scale, t);
          const bool qodd = (r + q_off) & 1;   // both query tiles start at a multiple of 128
          for (int i = 0; i < 3; ++i) {
            qt3[i] = qodd ? uint16_t(t[i] ^ 0x8000u) : t[i];   // the sign bit of f16 and bf16
            kt3[i] = (r & 1) ? to16<BF16>(-1.f) : one;
          }
        } else {   // the query side depends on the head: written per item by the producer
          for (int i = 0; i < 3; ++i) {
            qt3[i] = 0;
            kt3[i] = to16<BF16>(float(r) * (1.f / 128.f));
          }
        }
        for (int i = 0; i < 3; ++i) {
          *reinterpret_cast<uint16_t*>(sm.qaug + k16_offset(r, AUG_MOD + i)) = qt3[i];
          for (int st = 0; st < FWD_NST; ++st)
            *reinterpret_cast<uint16_t*>(sm.kaug[st] + k16_offset(r, AUG_MOD + i)) = kt3[i];
        }
      }
    }
    fence_async_smem();   // generic-proxy writes, read by the tensor core
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;

  if (warp == 0) {
    // ======================= producer: items, query tiles, K/V ring, per-stage columns =======================
    WC c{&sm.abort, p.status, p.timeout_ns, 1};
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
    }
    int last_u[FWD_NST];
    for (int s = 0; s < FWD_NST; ++s) last_u[s] = -1;
    int u = 0, last_q[2] = {-1, -1};
    bool ok = true;
    for (int ci = 0; ok; ++ci) {
      const int sl = ci & 1;
      int L = 0;
      if (lane == 0) L = persistent ? (int)atomicAdd(p.items, 1u) : (ci == 0 ? (int)(blockIdx.x % n_items) : n_claims);
      L = __shfl_sync(0xffffffffu, L, 0);
      // the slot's previous item (ci - 2) is done with everywhere
      if (ci >= 2 && !wait_warp(smem_u32(&sm.item_free[sl]), ((ci - 2) >> 1) & 1, c)) break;
      if (L >= n_claims) {   // no more items: the others stop at this slot
        if (lane == 0) {
          sm.item[sl] = -1;
          mbar_arrive(smem_u32(&sm.item_ready[sl]));
        }
        break;
      }
      const Item it = item_of(L);
      const long long dmi = (long long)it.b * p.dm.mb + (long long)it.h * p.dm.mh;   // dense-mask index of (b, h)
      for (int kb = lane; kb < p.nkb; kb += 32) {
        const int ks = p.km ? key_block_summary(p.km, it.b, p.Skv, kb) : p.km_sum ? p.km_sum[it.b * p.nkb + kb] : 2;
        for (int t = 0; t < 2; ++t) {
          const int qt = t ? it.qt1 : it.qt0;
          uint8_t f = 0;
          if (qt < p.nqb && ks != 0 && kb >= kb_lo && kb < kb_hi) {
            const int st =
                p.bm_tiles ? p.bm_tiles[it.b * p.bm_sb + it.h * p.bm_sh + (long long)qt * p.nkb + kb] : TILE_FULL;
            int ds = TILE_FULL;   // dense tile state: dense build only
            if constexpr (DM) ds = p.dm.tiles[(dmi * p.nqb + qt) * p.nkb + kb];
            if (st != TILE_EMPTY && ds != TILE_EMPTY)
              f = KB_VISIT | (st == TILE_PARTIAL && p.bm_mod != MASKMOD_NONE ? KB_MASKMOD : 0) |
                  (ks == 1 ? KB_KEYMASK : 0) | (ds == TILE_PARTIAL ? KB_DENSE : 0);
          }
          sm.flags[sl][t][kb] = f;
        }
      }
      if (lane == 0) {
        sm.item[sl] = L;
        if (MOD == MOD_ALIBI && fold) {
          // the item's head in the query side of the folded ALiBi term: columns
          // AUG_MOD .. +2 and AUG_KEY (the key mask's constant one) of a row are 8
          // contiguous bytes (the rest of the slot stays zero).  (One thread at
          // fixed offsets: stores from every lane of the producer cost the kernel
          // registers.)
          static_assert(AUG_MOD == 0 && AUG_KEY == 3, "one 8-byte store per query row");
          uint16_t t3[3];
          split3_plain<BF16>(128.f * exp2f(-8.0f * float(it.h + 1) / float(p.H)) * p.inv_scale, t3);
          const uint2 w = make_uint2(uint32_t(t3[0]) | (uint32_t(t3[1]) << 16),
                                     uint32_t(t3[2]) | (uint32_t(to16<BF16>(1.f)) << 16));
#pragma unroll
          for (int r = 0; r < 8; ++r) *reinterpret_cast<uint2*>(sm.qaug_h[sl] + k16_offset(r, 0)) = w;
          fence_async_smem();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.item_ready[sl]));   // release: the slot is visible to its waiters
      // the item's query tiles, into the slot's buffers (the S products of the
      // slot's previous item, which read them, were complete before item_free)
      if (lane == 0) {
        const uint32_t qbar = smem_u32(&sm.qfull[sl]);
        mbar_expect_tx(qbar, (it.valid1 ? 2 : 1) * FWD_TILE_BYTES);
        tma_load_2d(smem_u32(sm.q[sl][0]), &p.tm_q, qbar, 0, it.bh * p.Sq + it.qt0 * 128);
        if (it.valid1) tma_load_2d(smem_u32(sm.q[sl][1]), &p.tm_q, qbar, 0, it.bh * p.Sq + it.qt1 * 128);
      }
      last_q[sl] = ci;
      const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(it.h, p.H) : 0.f;
      for (int kb = 0; kb < p.nkb; ++kb) {
        const uint8_t fu = sm.flags[sl][0][kb] | sm.flags[sl][1][kb];
        if (!(fu & KB_VISIT)) continue;
        const int s = u % FWD_NST;
        // the block's key bits do not depend on the stage: their load is issued
        // before the wait for it, so its latency overlaps that wait
        uint32_t kbits = 0xffffffffu;
        if (kmask && (fu & KB_KEYMASK) && (aug || use_table)) kbits = lane_key_bits(p, it.b, kb * 128 + 4 * lane);
        if (u >= FWD_NST && !wait_warp(smem_u32(&sm.empty[s]), ((u / FWD_NST) - 1) & 1, c)) {
          ok = false;
          break;
        }
        if (aug) {
          if (kmask) {
            // lane owns keys 4 lane .. 4 lane + 3 of this kv block: column AUG_KEY of kaug[s]
            const uint32_t bits = kbits;
            // the infinity whose product with the scale is -inf (scale != 0)
            const uint16_t ninf = p.sc < 0.f ? (BF16 ? 0x7F80u : 0x7C00u) : (BF16 ? 0xFF80u : 0xFC00u);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int col = 4 * lane + i;
              *reinterpret_cast<uint16_t*>(sm.kaug[s] + k16_offset(col, AUG_KEY)) =
                  ((bits >> (col & 31)) & 1u) ? uint16_t(0) : ninf;
            }
          }
          fence_async_smem();
        } else if (use_table) {
          // lane owns columns 4 lane .. 4 lane + 3 of this kv block
          const uint32_t bits = kbits;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int col = 4 * lane + i;
            float base = ((bits >> (col & 31)) & 1u) ? 0.f : -INFINITY;
            if constexpr (MOD == MOD_ALIBI) base += slope2 * float(col);
            float e = base, o = base;
            if constexpr (MOD == MOD_CHECKER) {
              const float hb = (col & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;   // row parity 0
              e = base + hb;
              o = base - hb;
            }
            sm.cb[s][0][col] = e;
            sm.cb[s][1][col] = o;
          }
        }
        __syncwarp();
        // test hook: withhold the first copy so the consumers' bounded waits run out
        const bool withhold = p.inject_stall && u == 0;
        if (lane == 0 && !withhold) {
          const uint32_t fb = smem_u32(&sm.full[s]);
          mbar_expect_tx(fb, 2 * FWD_TILE_BYTES);   // release: the columns above are visible to its waiters
          tma_load_2d(smem_u32(sm.k[s]), &p.tm_k, fb, 0, it.bh * p.Skv + kb * 128);
          tma_load_2d(smem_u32(sm.v[s]), &p.tm_v, fb, 0, it.bh * p.Skv + kb * 128);
        }
        if (!withhold) last_u[s] = u;
        ++u;
      }
    }
    if (lane == 0) {   // every copy issued has landed before the CTA exits (instant unless aborted)
      for (int t = 0; t < 2; ++t)
        if (last_q[t] >= 0) drain_wait(smem_u32(&sm.qfull[t]), (last_q[t] >> 1) & 1, p.timeout_ns);
      for (int s = 0; s < FWD_NST; ++s)
        if (last_u[s] >= 0) drain_wait(smem_u32(&sm.full[s]), (last_u[s] / FWD_NST) & 1, p.timeout_ns);
    }
    __syncwarp();
  } else if (warp == 1 || warp == 2) {
    // ======================= MMA issue, one thread per tile =======================
    // Tile t's S_t(n+1) is issued as soon as its softmax has S_t(n) in registers
    // (sfree), so the product overlaps the exponentials; P_t(n) V goes out when
    // P_t(n) is in TMEM (pready).  Each tile arrives once per kv block on the
    // stage's empty barrier: a commit after its P V, or a plain arrival for a
    // block it skips.
    // Both threads run every item (a tile past the last query tile visits no
    // block but still arrives); the first P V of an item overwrites O.
    const int t = warp - 1;
    if (lane == 0) {
      WC c{&sm.abort, p.status, p.timeout_ns, 2 + 16 * t};
      constexpr uint32_t IDESC_S = idesc_f16(128, 128, BF16, false, false);
      constexpr uint32_t IDESC_PV = idesc_f16(128, 64, BF16, false, true);
      const uint32_t tS = tmem + 256 * t, tP = tS + 128, tO = tS + 192;
      const uint64_t qad0 = sdesc_k16(smem_u32(sm.qaug));
      uint64_t dk_[FWD_NST], dv_[FWD_NST];
      for (int s = 0; s < FWD_NST; ++s) {
        dk_[s] = sdesc_sw128(smem_u32(sm.k[s]), 16, 1024);
        dv_[s] = sdesc_sw128(smem_u32(sm.v[s]), 8192, 1024);
      }
      uint32_t n = 0;        // S products issued for this tile, over all items
      uint32_t n0 = 0;       // ... before the current item
      int s_pend = -1;       // stage of the block whose P V is still to issue
      uint32_t j_pend = 0;   // that block's index among this tile's visited blocks
      bool ok = true;
      auto issue_pv = [&]() -> bool {   // P_t(j_pend) V (stage s_pend), then release the stage
        if (!wait_one(smem_u32(&sm.pready[t]), j_pend & 1, c)) return false;
        tc_fence_after();
        const uint64_t vd = dv_[s_pend];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tO, tP + kk * 8, vd + 128 * kk, IDESC_PV, (kk > 0 || j_pend > n0) ? 1u : 0u);
        tc_commit(smem_u32(&sm.odone[t]));
        tc_commit(smem_u32(&sm.empty[s_pend]));
        s_pend = -1;
        return true;
      };
      int u = 0;
      for (int ci = 0; ok; ++ci) {
        const int sl = ci & 1;
        if (!wait_one(smem_u32(&sm.item_ready[sl]), (ci >> 1) & 1, c)) break;
        if (sm.item[sl] < 0) break;
        if (!wait_one(smem_u32(&sm.qfull[sl]), (ci >> 1) & 1, c)) break;
        n0 = n;
        const uint64_t qd = sdesc_sw128(smem_u32(sm.q[sl][t]), 16, 1024);
        const uint64_t qad = (MOD == MOD_ALIBI && fold) ? sdesc_k16_rows8(smem_u32(sm.qaug_h[sl])) : qad0;
        for (int kb = 0; ok && kb < p.nkb; ++kb) {
          const uint8_t f = sm.flags[sl][t][kb];
          if (!((f | sm.flags[sl][t ^ 1][kb]) & KB_VISIT)) continue;
          const int s = u % FWD_NST;
          if (!(f & KB_VISIT)) {
            // not this tile's block: first let any pending P V go (its stage must not be held)
            if (s_pend >= 0 && !issue_pv()) { ok = false; break; }
            if (!wait_one(smem_u32(&sm.full[s]), (u / FWD_NST) & 1, c)) { ok = false; break; }
            mbar_arrive(smem_u32(&sm.empty[s]));
            ++u;
            continue;
          }
          if (!wait_one(smem_u32(&sm.full[s]), (u / FWD_NST) & 1, c)) { ok = false; break; }
          if (n > 0 && !wait_one(smem_u32(&sm.sfree[t]), (n - 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
          const uint64_t kd = dk_[s];
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) mma_ss(tS, qd + 2 * kk, kd + 2 * kk, IDESC_S, kk > 0 ? 1u : 0u);
          if (aug) mma_ss(tS, qad, sdesc_k16(smem_u32(sm.kaug[s])), IDESC_S, 1u);
          tc_commit(smem_u32(&sm.sfull[t]));
          if (s_pend >= 0 && !issue_pv()) { ok = false; break; }
          s_pend = s;
          j_pend = n++;
          ++u;
        }
        if (!ok) break;
        if (s_pend >= 0 && !issue_pv()) break;
        mbar_arrive(smem_u32(&sm.item_free[sl]));
      }
      // every MMA issued by this thread completes before the CTA lets go of TMEM
      tc_commit(smem_u32(&sm.fin[t]));
      drain_wait(smem_u32(&sm.fin[t]), 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // ======================= softmax warpgroups =======================
    const int t = (warp - 3) >> 2;
    const int quad = warp & 3;   // TMEM lanes [32 quad, 32 quad + 32)
    WC c{&sm.abort, p.status, p.timeout_ns, 3 + t};
    const uint32_t lane_off = static_cast<uint32_t>(32 * quad) << 16;
    const uint32_t tS = tmem + lane_off + 256 * t;
    const uint32_t tP = tS + 128, tO = tS + 192;
    const int row = 32 * quad + lane;
    const uint64_t scv = f2(p.sc, p.sc);
    // unscaled scores in the max pass (scale > 0 keeps the order of the maximum)
    const bool raw = !use_table && MOD != MOD_USER && p.sc > 0.f;
    uint32_t n = 0;   // blocks of this tile, over all items (the barriers' phases)
    int u = 0;        // blocks of the items' unions (the ring's stages)
    bool ok = true;
    for (int ci = 0; ok; ++ci) {
      const int sl = ci & 1;
      if (!wait_warp(smem_u32(&sm.item_ready[sl]), (ci >> 1) & 1, c)) break;
      const int L = sm.item[sl];
      if (L < 0) break;
      const Item it = item_of(L);
      const int b = it.b, h = it.h, bh = it.bh;
      const int qt = t ? it.qt1 : it.qt0;
      if (qt >= p.nqb) {   // no rows of this tile in the item: the union's blocks only
        for (int kb = 0; kb < p.nkb; ++kb) u += ((sm.flags[sl][0][kb] | sm.flags[sl][1][kb]) & KB_VISIT) ? 1 : 0;
        mbar_arrive(smem_u32(&sm.item_free[sl]));
        continue;
      }
      const long long dmi = (long long)b * p.dm.mb + (long long)h * p.dm.mh;   // dense-mask index of (b, h)
      const int q = qt * 128 + row;
      const int qpos = q + q_off;   // the row's position among the keys (score mods, causal rule)
      const bool writer = quad == 3 && lane == 0;   // first warp of the group (warp 3 or 7)
      // the split variant's chunk of queries may end inside the tile: a warp whose
      // 32 rows all lie past Sq does no arithmetic, only the group's arrivals
      const bool idle = CHUNK && qt * 128 + 32 * quad >= p.Sq;
      const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
      const int parity = (MOD == MOD_CHECKER) ? (qpos & 1) : 0;
      float m_run = -INFINITY, l = 0.f;
      const uint32_t n0 = n;   // this item's first block of the tile
      for (int kb = 0; kb < p.nkb; ++kb) {
        const uint8_t f = sm.flags[sl][t][kb];
        const bool in_union = (f | sm.flags[sl][t ^ 1][kb]) & KB_VISIT;
        if (p.visited && writer)
          p.visited[((size_t)bh * p.nqb + qt) * p.nkb + kb] = (f & KB_VISIT) ? 1 : 0;
        if (!(f & KB_VISIT)) {
          u += in_union ? 1 : 0;
          continue;
        }
        const int s = u % FWD_NST;
        ++u;
        // this row's dense-mask bits for the block, fetched before the wait hides the load
        bool dense = false;
        uint4 dw = make_uint4(0u, 0u, 0u, 0u);
        if constexpr (DM) {
          dense = f & KB_DENSE;
          if (dense && q < p.Sq)
            dw = __ldg(reinterpret_cast<const uint4*>(p.dm.rowbits + (dmi * p.Sq + q) * (4LL * p.nkb)) + kb);
        }
        // the block's mask constants, ahead of the wait (they do not depend on S)
        const int kv0 = kb * 128;
        const bool causal = (MOD == MOD_CAUSAL && kv0 + 127 > qt * 128 + q_off) ||
                            ((f & KB_MASKMOD) && p.bm_mod == MASKMOD_CAUSAL);
        // keep column cc iff cc <= lim: the causal limit and, in a partial last kv
        // block, the end of the keys
        const int kvlim = p.Skv - 1 - kv0;
        const bool limited = causal || kvlim < 127;
        const int lim = causal ? min(qpos - kv0, kvlim) : kvlim;
        const float* tb = sm.cb[s][parity];
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        if (!wait_warp(smem_u32(&sm.sfull[t]), n & 1, c)) { ok = false; break; }
        // the stage's bias table was written before its full barrier was armed
        if (use_table && !wait_warp(smem_u32(&sm.full[s]), ((u - 1) / FWD_NST) & 1, c)) { ok = false; break; }
        tc_fence_after();
        if (idle) {
          // the same arrivals in the same order as the rows that compute: S free,
          // then (after P_t(n-1) V) P ready; the P and O rows of these lanes are
          // never read into a written row
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.sfree[t]));
          if (n > 0) {
            if (!wait_warp(smem_u32(&sm.odone[t]), (n - 1) & 1, c)) { ok = false; break; }
            tc_fence_after();
          }
          tc_fence_before();
          mbar_arrive(smem_u32(&sm.pready[t]));
          ++n;
          continue;
        }
        // The scale / mask / maximum pass over the NCK columns from column c0k on
        // (the block's constants above are set before S is read).  One
        // straight-line copy of the pass per (table, causal) pair: a runtime test
        // inside the unrolled loop would cost instructions on every score (a block
        // with dense-mask bits always takes the limited copy too).
        constexpr int NCK = 128;
        auto pass = [&](uint32_t (&rc)[NCK], int c0k) {
          const uint4 dwk = dw;
          if (use_table) {
            if (DM && dense) scale_scores<NCK, true, true, DM>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
            else if (limited) scale_scores<NCK, true, true, false>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
            else scale_scores<NCK, true, false, false>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
          } else if constexpr (MOD == MOD_USER) {
            // a PARTIAL tile of a user mask_mod's block mask: the expression masks each entry
            const bool umask = (f & KB_MASKMOD) && p.bm_mod == MASKMOD_USER;
            if (umask) {
              if (limited) scale_scores<NCK, false, true, false, true, false, true>(rc, scv, tb + c0k, lim - c0k, dwk, mx, b, h, qpos, kv0 + c0k);
              else scale_scores<NCK, false, false, false, true, false, true>(rc, scv, tb + c0k, lim - c0k, dwk, mx, b, h, qpos, kv0 + c0k);
            } else if (DM && dense) {
              scale_scores<NCK, false, true, DM, true>(rc, scv, tb + c0k, lim - c0k, dwk, mx, b, h, qpos, kv0 + c0k);
            } else if (limited) {
              scale_scores<NCK, false, true, false, true>(rc, scv, tb + c0k, lim - c0k, dwk, mx, b, h, qpos, kv0 + c0k);
            } else {
              scale_scores<NCK, false, false, false, true>(rc, scv, tb + c0k, lim - c0k, dwk, mx, b, h, qpos, kv0 + c0k);
            }
          } else if (raw) {
            if (DM && dense) scale_scores<NCK, false, true, DM, false, true>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
            else if (limited) scale_scores<NCK, false, true, false, false, true>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
            else scale_scores<NCK, false, false, false, false, true>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
          } else {
            if (DM && dense) scale_scores<NCK, false, true, DM>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
            else if (limited) scale_scores<NCK, false, true, false>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
            else scale_scores<NCK, false, false, false>(rc, scv, tb + c0k, lim - c0k, dwk, mx);
          }
        };
        uint32_t r[128];
        tmem_ld128(tS, r);
        // S_t(n) is in registers: the MMA thread may compute S_t(n+1) over it now
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.sfree[t]));
        pass(r, 0);
        // ALiBi's per-row constant for this block, slope2 (kv0 - q), is kept out of the
        // per-score work: scores here are x' = x - base
        const float base = (MOD == MOD_ALIBI) ? slope2 * float(kv0 - qpos) : 0.f;
        const float mxs = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
        const float rowmax = (raw ? mxs * p.sc : mxs) + base;
        // stale running max: rescale O only when the max grows by more than 2^8
        float alpha = 1.f;
        bool resc = false;
        if (m_run == -INFINITY) {
          m_run = rowmax;   // O holds only zero rows so far
        } else if (rowmax > m_run + 8.f) {
          alpha = ex2(m_run - rowmax);
          m_run = rowmax;
          resc = true;
        }
        const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
        const uint64_t negm = f2(base - m_use, base - m_use);
        // x = s scale - m on the raw path; x' - m (exactly x' + negm) otherwise
        const uint64_t mulv = raw ? scv : f2(1.f, 1.f);
        uint64_t sumv[2] = {f2(0.f, 0.f), f2(0.f, 0.f)};
        uint32_t pk[64];
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          float d0, d1;
          unf2(ffma2(f2(__uint_as_float(r[2 * i]), __uint_as_float(r[2 * i + 1])), mulv, negm), d0, d1);
          const float p0 = ex2(d0), p1 = ex2(d1);
          sumv[i & 1] = fadd2(sumv[i & 1], f2(p0, p1));
          pk[i] = pack2<BF16>(p0, p1);
        }
        // P_t(n-1) V must be done with the P region (and with O, if it is rescaled)
        if (n > 0) {
          if (!wait_warp(smem_u32(&sm.odone[t]), (n - 1) & 1, c)) { ok = false; break; }
          tc_fence_after();
        }
        tmem_st64(tP, pk);
        if (__any_sync(0xffffffffu, resc)) {
          uint32_t o[64];
          tmem_ld64(tO, o);
          const uint64_t av = f2(alpha, alpha);
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            float a0, a1;
            unf2(fmul2(f2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), av), a0, a1);
            o[2 * i] = __float_as_uint(a0);
            o[2 * i + 1] = __float_as_uint(a1);
          }
          tmem_st64(tO, o);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(smem_u32(&sm.pready[t]));
        float s0, s1, s2, s3;
        unf2(sumv[0], s0, s1);
        unf2(sumv[1], s2, s3);
        l = l * alpha + ((s0 + s1) + (s2 + s3));
        ++n;
      }
      tmem_st_wait();
      if (ok && n > n0) {
        if (!wait_warp(smem_u32(&sm.odone[t]), (n - 1) & 1, c))
          ok = false;
        else
          tc_fence_after();
      }
      if (ok) {
        const float inv = l > 0.f ? 1.f / l : 0.f;
        uint32_t o[64], w[32];
        if (n > n0) {
          tmem_ld64(tO, o);
        } else {
#pragma unroll
          for (int i = 0; i < 64; ++i) o[i] = 0u;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i)
          w[i] = pack2<BF16>(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
        // rows past Sq (partial last q tile) are computed, not written; the TMEM
        // load above stays warp-wide (tcgen05.ld is .sync.aligned)
        if (CHUNK && p.part && q < p.Sq) {
          // one kv range of a split: the unnormalised row, merged by launch_split_merge
          float* dst = p.part + (((size_t)bh * p.nsplit + split) * p.Sq + q) * FWD_PART;
          *reinterpret_cast<float4*>(dst) = make_float4(l > 0.f ? m_run : -INFINITY, l, 0.f, 0.f);
          uint4* od = reinterpret_cast<uint4*>(dst + 4);
#pragma unroll
          for (int i = 0; i < 16; ++i) od[i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
        } else if (q < p.Sq) {
          uint4* dst = reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(p.out) + ((size_t)bh * p.Sq + q) * 64);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
          const float m_fin = (m_run == -INFINITY) ? 0.f : m_run;
          p.lse[(size_t)bh * p.Sq + q] = l > 0.f ? (m_fin + lg2(l)) * kLn2 : -INFINITY;
        }
      }
      if (!ok) break;
      // the epilogue has read O out (its TMEM load waits): the next item's first P V may overwrite it
      tc_fence_before();
      mbar_arrive(smem_u32(&sm.item_free[sl]));
    }
  }

  // ---- teardown: all tcgen05 traffic of this CTA is finished before TMEM is freed
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

// ---------------------------------------------------------------------------
// host-side launcher
// ---------------------------------------------------------------------------
#ifndef __CUDACC_RTC__
size_t fwd_d64_smem_bytes() { return sizeof(FwdSmem) + 1024; }

// A forward kernel of this layout built elsewhere (a run-time-compiled score_mod):
// the same shared memory, grid and block as the built-in variants.
cudaError_t launch_fwd_d64_kernel(const FwdParams& p, const void* kern, cudaStream_t st) {
  const size_t smem = fwd_d64_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const unsigned grid = (unsigned)(p.items ? p.ctas : p.npairs * p.B * p.H * p.nsplit);
  void* args[] = {const_cast<FwdParams*>(&p)};
  return cudaLaunchKernel(kern, dim3(grid), dim3(FWD_THREADS), args, smem, st);
}

template <bool BF16, int MOD>
static cudaError_t launch_fwd_t(const FwdParams& p, cudaStream_t st) {
  const bool chunk = p.nsplit > 1 || p.q_off != 0;
  auto kern = chunk         ? fwd_d64_kernel<BF16, MOD, FWD_CHUNK>
              : p.dm.tiles ? fwd_d64_kernel<BF16, MOD, FWD_DENSE>
                           : fwd_d64_kernel<BF16, MOD, FWD_PLAIN>;
  const size_t smem = fwd_d64_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.items && !chunk ? p.ctas : p.npairs * p.B * p.H * p.nsplit));
  cfg.blockDim = dim3(FWD_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = chunk ? 1 : 0;   // the split variant waits itself
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}
#endif  // host

// One warp per row: M = max_s m_s, L = sum_s l_s 2^(m_s - M),
// O = sum_s O_s 2^(m_s - M) / L, lse = (M + log2 L) ln 2 (O = 0, lse = -inf
// when no split kept a key).  Lane j owns columns 2 j, 2 j + 1.
template <bool BF16>
__global__ void __launch_bounds__(256) split_merge_kernel(const float* __restrict__ part, int nsplit, long long rows,
                                                          int Sq, void* __restrict__ out, float* __restrict__ lse) {
  // launched with programmatic dependent launch behind the split forward: the
  // partial rows are read only once that grid has completed
  griddep_launch_dependents();
  griddep_wait();
  const long long r = blockIdx.x * 8LL + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  const long long bh = r / Sq, q = r % Sq;
  const float* base = part + ((size_t)bh * nsplit * Sq + q) * FWD_PART;
  const size_t stride = (size_t)Sq * FWD_PART;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, base[s * stride]);
  float Lsum = 0.f, o0 = 0.f, o1 = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < nsplit; ++s) {
      const float* ps = base + s * stride;
      const float m = ps[0];
      if (m == -INFINITY) continue;
      const float w = ex2(m - M);
      Lsum = fmaf(w, ps[1], Lsum);
      const float2 ov = *reinterpret_cast<const float2*>(ps + 4 + 2 * lane);
      o0 = fmaf(w, ov.x, o0);
      o1 = fmaf(w, ov.y, o1);
    }
  }
  const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
  reinterpret_cast<uint32_t*>(out)[r * 32 + lane] = pack2<BF16>(o0 * inv, o1 * inv);
  if (lane == 0) lse[r] = Lsum > 0.f ? (M + lg2(Lsum)) * kLn2 : -INFINITY;
}

#ifndef __CUDACC_RTC__
cudaError_t launch_split_merge(const float* part, int nsplit, long long rows, int Sq, void* out, float* lse, bool bf16,
                               cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + 7) / 8));
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return bf16 ? cudaLaunchKernelEx(&cfg, split_merge_kernel<true>, part, nsplit, rows, Sq, out, lse)
              : cudaLaunchKernelEx(&cfg, split_merge_kernel<false>, part, nsplit, rows, Sq, out, lse);
}

cudaError_t launch_fwd_d64(const FwdParams& p, bool bf16, int mod, cudaStream_t st) {
  if (bf16) {
    switch (mod) {
      case MOD_NONE: return launch_fwd_t<true, MOD_NONE>(p, st);
      case MOD_ALIBI: return launch_fwd_t<true, MOD_ALIBI>(p, st);
      case MOD_CHECKER: return launch_fwd_t<true, MOD_CHECKER>(p, st);
      default: return launch_fwd_t<true, MOD_CAUSAL>(p, st);
    }
  }
  switch (mod) {
    case MOD_NONE: return launch_fwd_t<false, MOD_NONE>(p, st);
    case MOD_ALIBI: return launch_fwd_t<false, MOD_ALIBI>(p, st);
    case MOD_CHECKER: return launch_fwd_t<false, MOD_CHECKER>(p, st);
    default: return launch_fwd_t<false, MOD_CAUSAL>(p, st);
  }
}

#endif  // host

}  // namespace attn
