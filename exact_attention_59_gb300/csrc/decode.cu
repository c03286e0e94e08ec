// decode.cu - single-query attention (q_len = 1), split-KV, HBM-bound.
//
// The flaxattention README ("Decoding", query length 1) times this case and
// lists "faster decoding attention" as a TODO; it is a streaming read of K and
// V, so the kernel is shaped for bandwidth, not for the tensor core:
//   grid (nsplit, B*H); each CTA takes a contiguous range of keys of one
//   (b, h); 8 lanes share one 128-byte key row (one 16-byte non-caching load
//   each), 4 rows per warp per step, 4 steps unrolled so every thread has
//   8 independent 16-byte loads in flight;
//   each 8-lane group runs its own online softmax (m, l, o[64] spread 8 per
//   lane), groups are merged in shared memory, and the CTA's (m, l, o) goes to
//   the workspace;
//   the last CTA of a (b, h) to finish (atomic ticket) merges the splits in a
//   fixed order, writes out and lse, and re-arms the ticket for the next call.
#include "kernels.h"

namespace attn {

constexpr int DEC_THREADS = 128;
constexpr int DEC_GROUPS = DEC_THREADS / 8;   // 16 key rows per step
constexpr int DEC_UNROLL = 4;

DEVI uint4 ld_stream(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <bool BF16>
DEVI void unpack8(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 t = unpack2<BF16>(w[i]);
    f[2 * i] = t.x;
    f[2 * i + 1] = t.y;
  }
}

int decode_num_splits(int B, int H, int Skv) {
  // aim for >= 4 CTAs per SM on 152 SMs, at least 64 keys per split
  const int bh = B * H;
  int ns = (4 * 152 + bh - 1) / bh;
  const int max_ns = (Skv + 63) / 64;
  if (ns > max_ns) ns = max_ns;
  if (ns < 1) ns = 1;
  return ns;
}

template <bool BF16, int MOD>
__global__ void __launch_bounds__(DEC_THREADS) decode_kernel(const DecodeParams p) {
  const int split = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int tid = threadIdx.x, grp = tid >> 3, part = tid & 7;
  const int k_lo = split * p.keys_per_split;
  const int k_hi = min(p.Skv, k_lo + p.keys_per_split);

  const uint16_t* qp = reinterpret_cast<const uint16_t*>(p.q) + (size_t)bh * 64 + part * 8;
  float qf[8];
  unpack8<BF16>(*reinterpret_cast<const uint4*>(qp), qf);
#pragma unroll
  for (int i = 0; i < 8; ++i) qf[i] *= p.sc;   // scale * log2(e) folded into q
  const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;

  const uint16_t* kbase = reinterpret_cast<const uint16_t*>(p.k) + (size_t)bh * p.Skv * 64 + part * 8;
  const uint16_t* vbase = reinterpret_cast<const uint16_t*>(p.v) + (size_t)bh * p.Skv * 64 + part * 8;
  const uint8_t* km = p.key_mask ? p.key_mask + (size_t)b * p.Skv : nullptr;

  float m = -INFINITY, l = 0.f, o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = 0.f;

  // The trip count and every shuffle are uniform across the CTA; keys past
  // the split's end are loaded by no one and contribute nothing.
  for (int jb = k_lo; jb < k_hi; jb += DEC_GROUPS * DEC_UNROLL) {
    uint4 kr[DEC_UNROLL], vr[DEC_UNROLL];
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
      const int j = jb + u * DEC_GROUPS + grp;
      if (j < k_hi) {
        kr[u] = ld_stream(kbase + (size_t)j * 64);
        vr[u] = ld_stream(vbase + (size_t)j * 64);
      } else {
        kr[u] = make_uint4(0u, 0u, 0u, 0u);
        vr[u] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int u = 0; u < DEC_UNROLL; ++u) {
      const int j = jb + u * DEC_GROUPS + grp;
      float kf[8];
      unpack8<BF16>(kr[u], kf);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) s = fmaf(qf[i], kf[i], s);
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      if (j >= k_hi) continue;
      if constexpr (MOD == MOD_ALIBI) s = fmaf(slope2, float(j), s);   // q_idx = 0
      if constexpr (MOD == MOD_CHECKER) s += (j & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;
      if constexpr (MOD == MOD_CAUSAL) if (j > 0) s = -INFINITY;
      if (km && km[j] == 0) s = -INFINITY;
      const float m_new = fmaxf(m, s);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m - m_use);
      const float pj = ex2(s - m_use);
      float vf[8];
      unpack8<BF16>(vr[u], vf);
#pragma unroll
      for (int i = 0; i < 8; ++i) o[i] = fmaf(pj, vf[i], o[i] * alpha);
      l = fmaf(l, alpha, pj);
      m = m_new;
    }
  }

  // ---- merge the 16 groups of this CTA
  __shared__ float sm_m[DEC_GROUPS], sm_l[DEC_GROUPS], sm_o[DEC_GROUPS][64];
  if (part == 0) {
    sm_m[grp] = m;
    sm_l[grp] = l;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) sm_o[grp][part * 8 + i] = o[i];
  __syncthreads();
  float* mine = p.partial + ((size_t)bh * p.nsplit + split) * (2 + 64);
  if (tid < 64) {
    float M = -INFINITY;
    for (int g = 0; g < DEC_GROUPS; ++g) M = fmaxf(M, sm_m[g]);
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Lsum = 0.f, acc = 0.f;
    for (int g = 0; g < DEC_GROUPS; ++g) {
      const float w = ex2(sm_m[g] - Mu);
      Lsum = fmaf(sm_l[g], w, Lsum);
      acc = fmaf(sm_o[g][tid], w, acc);
    }
    mine[2 + tid] = acc;
    if (tid == 0) {
      mine[0] = M;
      mine[1] = Lsum;
    }
  }
  // ---- the last CTA of this (b, h) merges all splits
  __shared__ unsigned ticket;
  __threadfence();
  __syncthreads();
  if (tid == 0) ticket = atomicAdd(p.counter + bh, 1u);
  __syncthreads();
  if (ticket != (unsigned)(p.nsplit - 1)) return;
  __threadfence();
  if (tid < 64) {
    const float* all = p.partial + (size_t)bh * p.nsplit * (2 + 64);
    float M = -INFINITY;
    for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, __ldcg(all + s * 66));
    const float Mu = (M == -INFINITY) ? 0.f : M;
    float Lsum = 0.f, acc = 0.f;
    for (int s = 0; s < p.nsplit; ++s) {
      const float w = ex2(__ldcg(all + s * 66) - Mu);
      Lsum = fmaf(__ldcg(all + s * 66 + 1), w, Lsum);
      acc = fmaf(__ldcg(all + s * 66 + 2 + tid), w, acc);
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    const float val = acc * inv;
    // pack pairs: even lanes write two outputs
    const float nb = __shfl_down_sync(0xffffffffu, val, 1);
    if ((tid & 1) == 0) {
      uint32_t* op = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + (size_t)bh * 64 + tid);
      *op = pack2<BF16>(val, nb);
    }
    if (tid == 0) {
      p.lse[bh] = Lsum > 0.f ? (Mu + lg2(Lsum)) * kLn2 : -INFINITY;
      p.counter[bh] = 0u;   // re-arm for the next call
    }
  }
}

template <bool BF16>
static cudaError_t launch_decode_t(const DecodeParams& p, cudaStream_t st) {
  dim3 grid(p.nsplit, p.B * p.H);
  switch (p.mod) {
    case MOD_NONE: decode_kernel<BF16, MOD_NONE><<<grid, DEC_THREADS, 0, st>>>(p); break;
    case MOD_ALIBI: decode_kernel<BF16, MOD_ALIBI><<<grid, DEC_THREADS, 0, st>>>(p); break;
    case MOD_CHECKER: decode_kernel<BF16, MOD_CHECKER><<<grid, DEC_THREADS, 0, st>>>(p); break;
    default: decode_kernel<BF16, MOD_CAUSAL><<<grid, DEC_THREADS, 0, st>>>(p); break;
  }
  return cudaGetLastError();
}

cudaError_t launch_decode(const DecodeParams& p, bool bf16, cudaStream_t st) {
  return bf16 ? launch_decode_t<true>(p, st) : launch_decode_t<false>(p, st);
}

}  // namespace attn
