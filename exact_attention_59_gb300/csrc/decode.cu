// decode.cu - single-query attention (q_len = 1), split-KV, HBM-bound.
//
// The flaxattention README ("Benchmark", decoding with query length 1) times
// this case and puts a faster decode on its to-do list ("Issues / TODO").  It
// is a streaming read of K and V (256 bytes per key at D = 64), so the kernel
// is shaped for bandwidth and latency, not for the tensor core:
//   one CTA per (b, h, split), each owning a contiguous range of up to
//   rounds x DEC_KEYS keys of one (b, h), walked in `rounds` rounds of
//   DEC_KEYS keys (128), DEC_WARP_KEYS per warp and round.  The launcher
//   takes the fewest rounds (a power of two up to DEC_ROUNDS_MAX) that let
//   every CTA of the call be resident at once, else the most.
//   Inside a warp, lane = 8 g + c: the lane group g (0..3) owns keys 4 u + g
//   (u < DEC_U) of the warp's share of the round and lane c of the group owns
//   head dimensions 8 c .. 8 c + 7.  Every lane issues all of its 16-byte K and
//   V loads of a round (ld.global.nc, no L1 allocation) before it uses any of
//   them: 32 KB in flight per CTA; consecutive lanes read consecutive 16-byte
//   pieces of the key rows, so every load instruction reads 512 contiguous
//   bytes.  The CTA asks L2 for its first DEC_PF_ROUNDS rounds of rows at
//   entry and for round r + DEC_PF_ROUNDS at the start of round r, so the rounds
//   after the first find their rows in L2 (at most 128 KB asked ahead per CTA).  Per round and lane group: the score of
//   each key (an 8-wide dot product, summed over the 8 lanes by three xor
//   shuffles), the mods and masks, and the exponentials and p-weighted sums of
//   V rows, merged into the group's running (m, l, o) by rescaling with
//   2^(m_old - m_new); then the groups and the warps are merged the same way.
//   With 512 threads and at most 64 registers a thread, two CTAs fit an SM:
//   the 256 CTAs of a 64-head, 2048-key call (4 rounds) run as one wave.
// The splits of a (b, h) form thread-block clusters of up to DEC_CLUSTER_MAX
// CTAs.  Each CTA stores its (m, l, o[64]) into the shared memory of the
// cluster's first CTA (distributed shared memory), one cluster barrier later
// that CTA merges them in rank order: no global-memory round trip.  A (b, h)
// with more splits than one cluster holds has several clusters; their first
// CTAs write (m, l, o) to the workspace and the last of them to finish
// (atomic ticket, zeroed by the launcher, no spin) merges those in a fixed order.
// Launched with programmatic dependent launch: a CTA first asks L2 for its
// first K and V rows, lets the next grid in the stream launch, and only then waits
// for the grids before it (griddepcontrol.wait).  Every load into registers
// (q, K, V, the key mask) and every store comes after that wait, so the
// stream-order contract is that of a plain launch: L2 is the GPU's point of
// coherence, so a line it fetched early still reflects writes made before the
// wait.  Back to back, one call's HBM stream overlaps the previous call's
// merge and drain.
// Arithmetic in base 2 (scale and biases carry log2(e)), as in the prefill.
#include "kernels.h"

namespace attn {

#ifndef ATTN_DEC_WARPS
#define ATTN_DEC_WARPS 16
#endif
#ifndef ATTN_DEC_U
#define ATTN_DEC_U 2
#endif
#ifndef ATTN_DEC_PDL
#define ATTN_DEC_PDL 1
#endif
#ifndef ATTN_DEC_ROUNDS   // DEC_KEYS-key rounds per CTA at most, one after the other in the same registers
#define ATTN_DEC_ROUNDS 16
#endif
#ifndef ATTN_DEC_CLUSTER_MAX   // CTAs per cluster at most (above 8 needs the non-portable size)
#define ATTN_DEC_CLUSTER_MAX 8
#endif
#ifndef ATTN_DEC_MINB   // resident CTAs per SM the register allocation must allow
#define ATTN_DEC_MINB (1024 / (32 * ATTN_DEC_WARPS) > 0 ? 1024 / (32 * ATTN_DEC_WARPS) : 1)
#endif
constexpr int DEC_WARPS = ATTN_DEC_WARPS;
constexpr int DEC_THREADS = 32 * DEC_WARPS;
constexpr int DEC_U = ATTN_DEC_U;                  // keys per lane group
constexpr int DEC_WARP_KEYS = 4 * DEC_U;           // keys per warp and round
constexpr int DEC_KEYS = DEC_WARPS * DEC_WARP_KEYS;   // keys per CTA and round
constexpr int DEC_CLUSTER_MAX = ATTN_DEC_CLUSTER_MAX;
constexpr int DEC_ROUNDS_MAX = ATTN_DEC_ROUNDS;
constexpr int DEC_PF_ROUNDS = 4;   // rounds of rows a CTA has asked L2 for ahead of its loads

int decode_num_splits(int B, int H, int Skv) {
  (void)B;
  (void)H;
  return (Skv + DEC_KEYS - 1) / DEC_KEYS;
}

// 16-byte read-only load that does not allocate in L1 (each byte is read once).
DEVI uint4 ldg_stream(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Merges the running (m, l, o) of this lane with the one `off` lanes away.
DEVI void merge_xor(float& m, float& l, float (&o)[8], int off) {
  const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
  const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
  const float M = fmaxf(m, m2);
  const float Mu = (M == -INFINITY) ? 0.f : M;
  const float a = ex2(m - Mu), b = ex2(m2 - Mu);   // 2^-inf = 0 for an empty side
  l = l * a + l2 * b;
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = o[e] * a + __shfl_xor_sync(0xffffffffu, o[e], off) * b;
  m = M;
}

template <bool BF16, int MOD>
__global__ void __launch_bounds__(DEC_THREADS, ATTN_DEC_MINB) decode_kernel(const DecodeParams p) {
  // blockIdx.x = (bh * ngroups + group) * cluster + rank; split = group * cluster + rank
  const int per_head = p.ngroups * p.cluster;
  const int bh = blockIdx.x / per_head, split = blockIdx.x % per_head;
  const int group = split / p.cluster;
  const uint32_t rank = cluster_ctarank();
  const int b = bh / p.H, h = bh % p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 3, c = lane & 7;
  const int k_lo = split * p.keys_per_split;             // may be >= Skv: an empty split
  const int k_hi = min(p.Skv, k_lo + p.keys_per_split);

  __shared__ float sm_m[DEC_WARPS], sm_l[DEC_WARPS], sm_o[DEC_WARPS][64];
  __shared__ float sm_part[DEC_CLUSTER_MAX][2 + 64];   // the cluster's CTAs' (m, l, o); read in rank 0
  __shared__ unsigned ticket;
  // the cluster's CTAs have all started before any writes into rank 0's shared
  // memory (the matching wait is just before those writes)
  cluster_arrive_relaxed();

  // (before the loads: the slope's exp2 then needs no registers beside them)
  const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
  // L2 prefetch of rounds [r0, r1) of this CTA's K (thread 0) and V (thread 1)
  // rows: contiguous, 128 bytes a row
  auto prefetch_rounds = [&](int r0, int r1) {
    const int a = k_lo + r0 * DEC_KEYS, e = min(k_hi, k_lo + r1 * DEC_KEYS);
    if (tid < 2 && e > a) {
      const size_t row0 = (size_t)bh * p.Skv + a;
      const unsigned char* base = static_cast<const unsigned char*>(tid == 0 ? p.k : p.v) + row0 * 128;
      prefetch_l2_bulk(base, static_cast<uint32_t>(e - a) * 128u);
    }
  };
  prefetch_rounds(0, DEC_PF_ROUNDS);
#if ATTN_DEC_PDL
  griddep_launch_dependents();
  griddep_wait();
#endif
  // q (this lane's 8 dimensions), scaled by scale * log2(e)
  float qf[8];
  {
    const uint4 qw = __ldg(reinterpret_cast<const uint4*>(p.q) + (size_t)bh * 8 + c);
    const uint32_t w4[4] = {qw.x, qw.y, qw.z, qw.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = unpack2<BF16>(w4[e]);
      qf[2 * e] = f.x * p.sc;
      qf[2 * e + 1] = f.y * p.sc;
    }
  }

  // ---- K and V of round rd: this lane's 16-byte pieces of its group's keys,
  // and the key mask's bytes (0 / 1 for out-of-range keys is settled later)
  const uint4* kg = reinterpret_cast<const uint4*>(p.k) + (size_t)bh * p.Skv * 8 + c;
  const uint4* vg = reinterpret_cast<const uint4*>(p.v) + (size_t)bh * p.Skv * 8 + c;
  auto issue_round = [&](int rd, uint4 (&kr)[DEC_U], uint4 (&vr)[DEC_U], uint32_t (&kb)[DEC_U]) {
    const int kw = k_lo + rd * DEC_KEYS + DEC_WARP_KEYS * warp;
#pragma unroll
    for (int u = 0; u < DEC_U; ++u) {
      const int key = kw + 4 * u + g;
      if (key < k_hi) {
        kr[u] = ldg_stream(kg + (size_t)key * 8);
        vr[u] = ldg_stream(vg + (size_t)key * 8);
        kb[u] = p.key_mask ? static_cast<uint32_t>(__ldg(p.key_mask + (size_t)b * p.Skv + key)) : 1u;
      } else {
        kr[u] = make_uint4(0u, 0u, 0u, 0u);
        vr[u] = make_uint4(0u, 0u, 0u, 0u);
        kb[u] = 0u;
      }
    }
  };
  // running (m, l, o) of this lane group over the rounds
  float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
  uint4 kr[DEC_U], vr[DEC_U];
  uint32_t kb[DEC_U];
  issue_round(0, kr, vr, kb);
#pragma unroll 1   // one round's loads in registers at a time
  for (int rd = 0; rd < p.rounds; ++rd) {
    // round rd: keys k_lo + rd DEC_KEYS + [DEC_WARP_KEYS warp, DEC_WARP_KEYS (warp + 1))
    const int kw = k_lo + rd * DEC_KEYS + DEC_WARP_KEYS * warp;
    prefetch_rounds(rd + DEC_PF_ROUNDS, rd + DEC_PF_ROUNDS + 1);   // rolling: DEC_PF_ROUNDS rounds ahead
    // ---- scores of the group's keys (partial dot over 8 dims, then over the 8 lanes)
    float s[DEC_U];
#pragma unroll
    for (int u = 0; u < DEC_U; ++u) {
      const uint32_t w4[4] = {kr[u].x, kr[u].y, kr[u].z, kr[u].w};
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack2<BF16>(w4[e]);
        acc = fmaf(qf[2 * e], f.x, acc);
        acc = fmaf(qf[2 * e + 1], f.y, acc);
      }
      s[u] = acc;
    }
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) {
#pragma unroll
      for (int u = 0; u < DEC_U; ++u) s[u] += __shfl_xor_sync(0xffffffffu, s[u], off);
    }
    float mr = -INFINITY;
#pragma unroll
    for (int u = 0; u < DEC_U; ++u) {
      const int kv = kw + 4 * u + g;   // q_idx = 0
      float x = s[u];
      if constexpr (MOD == MOD_ALIBI) x = fmaf(slope2, float(kv), x);
      if constexpr (MOD == MOD_CHECKER) x += (kv & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;
      if constexpr (MOD == MOD_CAUSAL) x = kv > 0 ? -INFINITY : x;
      x = kb[u] != 0u ? x : -INFINITY;   // in range and kept by the key mask
      s[u] = x;
      mr = fmaxf(mr, x);
    }
    // ---- exponentials and the p-weighted sum of V rows (this lane's 8 dims),
    // merged into the running (m, l, o) of the earlier rounds
    const float mn = fmaxf(m, mr);
    const float mu = (mn == -INFINITY) ? 0.f : mn;
    {
      const float a = ex2(m - mu);   // 0 while m = -inf
      l *= a;
#pragma unroll
      for (int e = 0; e < 8; ++e) o[e] *= a;
    }
    m = mn;
#pragma unroll
    for (int u = 0; u < DEC_U; ++u) {
      const float pu = ex2(s[u] - mu);
      l += pu;
      const uint32_t w4[4] = {vr[u].x, vr[u].y, vr[u].z, vr[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = unpack2<BF16>(w4[e]);
        o[2 * e] = fmaf(pu, f.x, o[2 * e]);
        o[2 * e + 1] = fmaf(pu, f.y, o[2 * e + 1]);
      }
    }
    if (rd + 1 < p.rounds) issue_round(rd + 1, kr, vr, kb);
  }
  // ---- the four lane groups of the warp, then the four warps of the CTA
  merge_xor(m, l, o, 8);
  merge_xor(m, l, o, 16);
  if (g == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) sm_o[warp][8 * c + e] = o[e];
    if (c == 0) {
      sm_m[warp] = m;
      sm_l[warp] = l;
    }
  }
  __syncthreads();
  // ---- this CTA's (m, l, o) into slot `rank` of the cluster's first CTA
  float cm = -INFINITY, cl = 0.f, co = 0.f;
  if (tid < 64) {
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) cm = fmaxf(cm, sm_m[w]);
    const float mu2 = (cm == -INFINITY) ? 0.f : cm;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float a = ex2(sm_m[w] - mu2);
      cl = fmaf(sm_l[w], a, cl);
      co = fmaf(sm_o[w][tid], a, co);
    }
  }
  cluster_wait_acquire();   // every CTA of the cluster is running
  if (tid < 64) {
    const uint32_t slot = mapa_shared(smem_u32(&sm_part[rank][0]), 0);
    st_cluster_f32(slot + 4u * (2 + tid), co);
    if (tid == 0) {
      st_cluster_f32(slot, cm);
      st_cluster_f32(slot + 4u, cl);
    }
  }
  cluster_arrive_release();
  cluster_wait_acquire();
  if (rank != 0) return;
  // ---- rank 0: merge the cluster's slots in rank order
  float M = -INFINITY, L = 0.f, O = 0.f;
  if (tid < 64) {
    for (int r = 0; r < p.cluster; ++r) M = fmaxf(M, sm_part[r][0]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    for (int r = 0; r < p.cluster; ++r) {
      const float a = ex2(sm_part[r][0] - Mu);
      L = fmaf(sm_part[r][1], a, L);
      O = fmaf(sm_part[r][2 + tid], a, O);
    }
  }
  if (p.ngroups == 1) {   // the whole (b, h) in one cluster
    if (tid < 64) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const float val = O * inv;
      const float nb = __shfl_down_sync(0xffffffffu, val, 1);
      if ((tid & 1) == 0) {
        uint32_t* op = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + (size_t)bh * 64 + tid);
        *op = pack2<BF16>(val, nb);
      }
      if (tid == 0) p.lse[bh] = L > 0.f ? (((M == -INFINITY) ? 0.f : M) + lg2(L)) * kLn2 : -INFINITY;
    }
    return;
  }
  // ---- several clusters per (b, h): partials through the workspace
  if (tid < 64) {
    float* mine = p.partial + ((size_t)bh * p.ngroups + group) * (2 + 64);
    mine[2 + tid] = O;
    if (tid == 0) {
      mine[0] = M;
      mine[1] = L;
    }
  }
  // The CTA barrier orders the partial's stores before thread 0's fence, whose
  // gpu-scope ordering covers them (cumulativity), so one fence per CTA
  // publishes the partial before its ticket.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    ticket = atomicAdd(p.counter + bh, 1u);
  }
  __syncthreads();
  if (ticket != (unsigned)(p.ngroups - 1)) return;
  if (tid == 0) __threadfence();
  __syncthreads();
  // max over the groups: threads stride over them, then a CTA reduction
  const float* all = p.partial + (size_t)bh * p.ngroups * (2 + 64);
  float Mx = -INFINITY;
  for (int sidx = tid; sidx < p.ngroups; sidx += DEC_THREADS) Mx = fmaxf(Mx, __ldcg(all + (size_t)sidx * 66));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
  if (lane == 0) sm_m[warp] = Mx;
  __syncthreads();
  Mx = sm_m[0];
#pragma unroll
  for (int w = 1; w < DEC_WARPS; ++w) Mx = fmaxf(Mx, sm_m[w]);
  const float Mxu = (Mx == -INFINITY) ? 0.f : Mx;
  // thread (part, d) sums dimension d over the groups congruent to part mod DEC_THREADS / 64
  const int d = tid & 63, part = tid >> 6;
  float Lsum = 0.f, acc = 0.f;
  for (int sidx = part; sidx < p.ngroups; sidx += DEC_THREADS / 64) {
    const float* ps = all + (size_t)sidx * 66;
    const float w = ex2(__ldcg(ps) - Mxu);
    Lsum = fmaf(__ldcg(ps + 1), w, Lsum);
    acc = fmaf(__ldcg(ps + 2 + d), w, acc);
  }
  __syncthreads();   // sm_o and sm_l are reused below
  if (part > 0) {
    sm_o[part][d] = acc;
    if (d == 0) sm_l[part] = Lsum;
  }
  __syncthreads();
  if (part == 0) {
#pragma unroll
    for (int j = 1; j < DEC_THREADS / 64; ++j) {   // fixed order
      acc += sm_o[j][d];
      Lsum += sm_l[j];
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    const float val = acc * inv;
    const float nb = __shfl_down_sync(0xffffffffu, val, 1);
    if ((d & 1) == 0) {
      uint32_t* op = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + (size_t)bh * 64 + d);
      *op = pack2<BF16>(val, nb);
    }
    if (d == 0) p.lse[bh] = Lsum > 0.f ? (Mxu + lg2(Lsum)) * kLn2 : -INFINITY;
  }
}

template <bool BF16, int MOD>
static cudaError_t launch_decode_k(const DecodeParams& p, cudaStream_t st) {
  auto kern = decode_kernel<BF16, MOD>;
  if (p.cluster > 8) {
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)p.B * p.H * p.ngroups * p.cluster));
  cfg.blockDim = dim3(DEC_THREADS);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = ATTN_DEC_PDL ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = (unsigned)p.cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <bool BF16>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t st) {
  switch (p.mod) {
    case MOD_NONE: return launch_decode_k<BF16, MOD_NONE>(p, st);
    case MOD_ALIBI: return launch_decode_k<BF16, MOD_ALIBI>(p, st);
    case MOD_CHECKER: return launch_decode_k<BF16, MOD_CHECKER>(p, st);
    default: return launch_decode_k<BF16, MOD_CAUSAL>(p, st);
  }
}

// p.nsplit: the workspace's split count (ceil(Skv / DEC_KEYS) rows of partials
// per (b, h)).  Here the rounds per CTA are the fewest powers of two up to
// DEC_ROUNDS_MAX that let all CTAs be resident at once (ATTN_DEC_MINB per
// SM), else the most; ceil(Skv / (DEC_KEYS rounds)) CTAs per (b, h) are
// grouped into clusters of at most DEC_CLUSTER_MAX, ngroups clusters per
// (b, h), and the keys spread evenly over ngroups x cluster CTAs (at most
// DEC_KEYS rounds each; ngroups <= nsplit, so the partials fit).
cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t st) {
  if (p.nsplit < 1 || p.Skv < 1 || p.keys_per_split > DEC_KEYS || p.keys_per_split < 1) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidDevice;
  const long long slots = (long long)sms * ATTN_DEC_MINB;
  const long long BH = (long long)p.B * p.H;
  DecodeParams q = p;
  q.rounds = 1;
  while (q.rounds < DEC_ROUNDS_MAX &&
         BH * ((p.Skv + (long long)DEC_KEYS * q.rounds - 1) / ((long long)DEC_KEYS * q.rounds)) > slots)
    q.rounds *= 2;
  if (q.rounds > DEC_ROUNDS_MAX) q.rounds = DEC_ROUNDS_MAX;
  const int want = (int)((p.Skv + (long long)DEC_KEYS * q.rounds - 1) / ((long long)DEC_KEYS * q.rounds));   // <= nsplit
  q.cluster = want < DEC_CLUSTER_MAX ? want : DEC_CLUSTER_MAX;
  q.ngroups = (want + q.cluster - 1) / q.cluster;
  const long long ctas_per_head = (long long)q.ngroups * q.cluster;
  q.keys_per_split = (int)((p.Skv + ctas_per_head - 1) / ctas_per_head);
  if (BH * ctas_per_head > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (q.ngroups > 1) {   // the clusters' tickets start at zero in every call
    const cudaError_t e = cudaMemsetAsync(q.counter, 0, (size_t)BH * sizeof(unsigned), st);
    if (e != cudaSuccess) return e;
  }
  return bf16 ? launch_decode_t<true>(q, st) : launch_decode_t<false>(q, st);
}

}  // namespace attn
