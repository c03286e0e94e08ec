// decode.cu - single-query attention (q_len = 1), split-KV, HBM-bound.
//
// The flaxattention README ("Decoding", query length 1) times this case and
// lists "faster decoding attention" as a TODO.  It is a streaming read of K and
// V (256 bytes per key at D = 64), so the kernel is shaped for bandwidth and
// latency, not for the tensor core:
//   one CTA per (b, h, split), the splits of a head adjacent; each CTA owns a contiguous range of up to DEC_KEYS keys
//   of one (b, h), DEC_WARP_KEYS per warp.  Inside a warp, lane = 8 g + c: the
//   lane group g (0..3) owns keys 4 u + g (u < DEC_U) of the warp's range and
//   lane c of the group owns head dimensions 8 c .. 8 c + 7.  Every lane issues
//   all of its 16-byte K and V loads (ld.global.nc, no L1 allocation) before it
//   uses any of them, so each CTA has 32 KB in flight at once and the HBM
//   latency is paid once per CTA; consecutive lanes read consecutive 16-byte
//   pieces of the key rows, so every load instruction reads 512 contiguous
//   bytes.  No shared-memory staging and no barrier wait: nothing can stall.
//   Per lane group: the score of each key (an 8-wide dot product, summed over
//   the 8 lanes by three xor shuffles), the mods and masks, a local max, the
//   exponentials and p-weighted sums of V rows; the groups and then the warps
//   are merged with the usual rescaling by 2^(m_i - M).  The CTA's (m, l, o[64])
//   goes to the workspace.
//   The last CTA of a (b, h) to finish (atomic ticket, no spin) merges the
//   splits in a fixed order, writes out and lse, and re-arms the ticket.
// Arithmetic in base 2 (scale and biases carry log2(e)), as in the prefill.
#include "kernels.h"

namespace attn {

#ifndef ATTN_DEC_WARPS
#define ATTN_DEC_WARPS 8
#endif
#ifndef ATTN_DEC_U
#define ATTN_DEC_U 4
#endif
constexpr int DEC_WARPS = ATTN_DEC_WARPS;
constexpr int DEC_THREADS = 32 * DEC_WARPS;
constexpr int DEC_U = ATTN_DEC_U;                  // keys per lane group
constexpr int DEC_WARP_KEYS = 4 * DEC_U;           // 16
constexpr int DEC_KEYS = DEC_WARPS * DEC_WARP_KEYS;   // 128 keys per CTA at most

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
__global__ void __launch_bounds__(DEC_THREADS, (1024 / DEC_THREADS > 0 ? 1024 / DEC_THREADS : 1)) decode_kernel(const DecodeParams p) {
  const int split = blockIdx.x % p.nsplit, bh = blockIdx.x / p.nsplit;
  const int b = bh / p.H, h = bh % p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 3, c = lane & 7;
  const int k_lo = split * p.keys_per_split;
  const int k_hi = min(p.Skv, k_lo + p.keys_per_split);
  const int kw = k_lo + DEC_WARP_KEYS * warp;   // first key of this warp

  __shared__ float sm_m[DEC_WARPS], sm_l[DEC_WARPS], sm_o[DEC_WARPS][64];
  __shared__ unsigned ticket;

  // (before the loads: the slope's exp2 then needs no registers beside them)
  const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
  // ---- every K and V load of this lane goes out first
  const uint4* kg = reinterpret_cast<const uint4*>(p.k) + (size_t)bh * p.Skv * 8 + c;
  const uint4* vg = reinterpret_cast<const uint4*>(p.v) + (size_t)bh * p.Skv * 8 + c;
  uint4 kr[DEC_U], vr[DEC_U];
#pragma unroll
  for (int u = 0; u < DEC_U; ++u) {
    const int key = kw + 4 * u + g;
    if (key < k_hi) {
      kr[u] = ldg_stream(kg + (size_t)key * 8);
      vr[u] = ldg_stream(vg + (size_t)key * 8);
    } else {
      kr[u] = make_uint4(0u, 0u, 0u, 0u);
      vr[u] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  uint32_t keep = 0;   // bit u: key 4 u + g of the warp's range is in range and kept
#pragma unroll
  for (int u = 0; u < DEC_U; ++u) {
    const int key = kw + 4 * u + g;
    const bool in = key < k_hi && (!p.key_mask || __ldg(p.key_mask + (size_t)b * p.Skv + key) != 0);
    keep |= (in ? 1u : 0u) << u;
  }
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
  float m = -INFINITY;
#pragma unroll
  for (int u = 0; u < DEC_U; ++u) {
    const int kv = kw + 4 * u + g;   // q_idx = 0
    float x = s[u];
    if constexpr (MOD == MOD_ALIBI) x = fmaf(slope2, float(kv), x);
    if constexpr (MOD == MOD_CHECKER) x += (kv & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;
    if constexpr (MOD == MOD_CAUSAL) x = kv > 0 ? -INFINITY : x;
    x = ((keep >> u) & 1u) ? x : -INFINITY;
    s[u] = x;
    m = fmaxf(m, x);
  }
  // ---- exponentials and the p-weighted sum of V rows (this lane's 8 dims)
  const float mu = (m == -INFINITY) ? 0.f : m;
  float l = 0.f, o[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) o[e] = 0.f;
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
  if (tid < 64) {
    float M = sm_m[0];
#pragma unroll
    for (int w = 1; w < DEC_WARPS; ++w) M = fmaxf(M, sm_m[w]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, O = 0.f;
#pragma unroll
    for (int w = 0; w < DEC_WARPS; ++w) {
      const float a = ex2(sm_m[w] - Mu);
      L = fmaf(sm_l[w], a, L);
      O = fmaf(sm_o[w][tid], a, O);
    }
    float* mine = p.partial + ((size_t)bh * p.nsplit + split) * (2 + 64);
    mine[2 + tid] = O;
    if (tid == 0) {
      mine[0] = M;
      mine[1] = L;
    }
  }
  // ---- the last CTA of this (b, h) merges all splits.  The CTA barrier orders the
  // partial's stores before thread 0's fence, whose gpu-scope ordering covers
  // them (cumulativity), so one fence per CTA publishes the partial before its ticket.
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    ticket = atomicAdd(p.counter + bh, 1u);
  }
  __syncthreads();
  if (ticket != (unsigned)(p.nsplit - 1)) return;
  if (tid == 0) __threadfence();
  __syncthreads();
  // max over the splits: threads stride over them, then a CTA reduction
  const float* all = p.partial + (size_t)bh * p.nsplit * (2 + 64);
  float Mx = -INFINITY;
  for (int sidx = tid; sidx < p.nsplit; sidx += DEC_THREADS) Mx = fmaxf(Mx, __ldcg(all + (size_t)sidx * 66));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) Mx = fmaxf(Mx, __shfl_xor_sync(0xffffffffu, Mx, off));
  if (lane == 0) sm_m[warp] = Mx;
  __syncthreads();
  Mx = sm_m[0];
#pragma unroll
  for (int w = 1; w < DEC_WARPS; ++w) Mx = fmaxf(Mx, sm_m[w]);
  const float Mxu = (Mx == -INFINITY) ? 0.f : Mx;
  // thread (part, d) sums dimension d over the splits congruent to part mod 4
  const int d = tid & 63, part = tid >> 6;
  float Lsum = 0.f, acc = 0.f;
  for (int sidx = part; sidx < p.nsplit; sidx += DEC_THREADS / 64) {
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
    if (d == 0) {
      p.lse[bh] = Lsum > 0.f ? (Mxu + lg2(Lsum)) * kLn2 : -INFINITY;
      p.counter[bh] = 0u;   // re-arm for the next call
    }
  }
}

template <bool BF16>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t st) {
  const long long n = (long long)p.nsplit * p.B * p.H;   // one CTA per (b, h, split), splits of a head adjacent
  if (n > 0x7fffffffLL) return cudaErrorInvalidValue;
  const unsigned grid = (unsigned)n;
  switch (p.mod) {
    case MOD_NONE: decode_kernel<BF16, MOD_NONE><<<grid, DEC_THREADS, 0, st>>>(p); break;
    case MOD_ALIBI: decode_kernel<BF16, MOD_ALIBI><<<grid, DEC_THREADS, 0, st>>>(p); break;
    case MOD_CHECKER: decode_kernel<BF16, MOD_CHECKER><<<grid, DEC_THREADS, 0, st>>>(p); break;
    default: decode_kernel<BF16, MOD_CAUSAL><<<grid, DEC_THREADS, 0, st>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t st) {
  if (p.keys_per_split > DEC_KEYS || p.keys_per_split < 1) return cudaErrorInvalidValue;
  return bf16 ? launch_decode_t<true>(p, st) : launch_decode_t<false>(p, st);
}

}  // namespace attn
