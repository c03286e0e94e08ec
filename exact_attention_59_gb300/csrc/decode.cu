// decode.cu - single-query attention (q_len = 1), split-KV, HBM-bound.
//
// The flaxattention README ("Decoding", query length 1) times this case and
// lists "faster decoding attention" as a TODO.  It is a streaming read of K and
// V (256 bytes per key at D = 64), so the kernel is shaped for bandwidth and
// latency, not for the tensor core:
//   grid (nsplit, B*H); each CTA owns a contiguous range of up to 128 keys of
//   one (b, h).  Its K and V rows are contiguous in HBM, so one thread issues
//   two bulk copies (cp.async.bulk, 16-byte aligned, 16 KB each) into shared
//   memory completing on one mbarrier: a single round trip to HBM per CTA.
//   At 33 KB of shared memory a CTA, 6 fit on an SM, so the B8 H8 Skv 2048
//   case runs 912 of its 1024 CTAs in the first wave (all of K and V, 33.5
//   MB, is more than the GPU's shared memory); streaming each split through a
//   two-stage ring instead, to fit one wave, was slower (a second round trip
//   per CTA).
//   In shared memory: thread j forms the score of key j, the CTA takes the max
//   and the exponentials, and thread d (and d + 64) sum p_j V_jd over half the
//   keys each; the CTA's (m, l, o[64]) goes to the workspace.
//   The last CTA of a (b, h) to finish (atomic ticket) merges the splits in a
//   fixed order, writes out and lse, and re-arms the ticket for the next call.
#include "kernels.h"

namespace attn {

constexpr int DEC_THREADS = 128;
constexpr int DEC_KEYS = 128;   // keys per split (maximum): 32 KB of K and V per CTA

int decode_num_splits(int B, int H, int Skv) {
  (void)B;
  (void)H;
  return (Skv + DEC_KEYS - 1) / DEC_KEYS;
}

DEVI void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
               : "memory");
}

template <bool BF16, int MOD>
__global__ void __launch_bounds__(DEC_THREADS) decode_kernel(const DecodeParams p) {
  const int split = blockIdx.x, bh = blockIdx.y;
  const int b = bh / p.H, h = bh % p.H;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int k_lo = split * p.keys_per_split;
  const int nk = min(p.Skv, k_lo + p.keys_per_split) - k_lo;   // 1 .. 128

  __shared__ __align__(128) uint16_t ks[DEC_KEYS * 64], vs[DEC_KEYS * 64];
  __shared__ __align__(16) float qs[64];
  __shared__ float sc_s[DEC_KEYS], redm[4], reds[4], o_part[64];
  __shared__ __align__(8) uint64_t bar;
  __shared__ unsigned ticket;

  const uint32_t barp = smem_u32(&bar);
  if (tid == 0) {
    mbar_init(barp, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint32_t bytes = (uint32_t)nk * 128u;
    mbar_expect_tx(barp, 2 * bytes);
    const uint16_t* kg = reinterpret_cast<const uint16_t*>(p.k) + ((size_t)bh * p.Skv + k_lo) * 64;
    const uint16_t* vg = reinterpret_cast<const uint16_t*>(p.v) + ((size_t)bh * p.Skv + k_lo) * 64;
    bulk_g2s(smem_u32(ks), kg, bytes, barp);
    bulk_g2s(smem_u32(vs), vg, bytes, barp);
  }
  // q (scaled by scale * log2 e) while the copies fly
  if (tid < 32) {
    const uint32_t w = reinterpret_cast<const uint32_t*>(p.q)[(size_t)bh * 32 + tid];
    const float2 f = unpack2<BF16>(w);
    qs[2 * tid] = f.x * p.sc;
    qs[2 * tid + 1] = f.y * p.sc;
  }
  const float slope2 = (MOD == MOD_ALIBI) ? alibi_slope_log2(h, p.H) : 0.f;
  // The copies complete in well under a millisecond; a generous bounded spin
  // keeps a lost completion from hanging the GPU (the status word records it).
  bool ok = true;
  {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(barp, 0)) {
      if (global_timer_ns() - t0 > 2000000000ull) { ok = false; break; }
    }
  }
  __syncthreads();

  // ---- scores: thread j owns key j (its 64 dims as eight 16-byte chunks, the
  // start rotated by j so the lanes of a warp spread over the banks)
  float x = -INFINITY;
  {
    const int j = tid;
    if (j < nk) {
      const uint4* kr = reinterpret_cast<const uint4*>(ks + j * 64);
      float s = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int c = (i + j) & 7;
        const uint4 u = kr[c];
        const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = unpack2<BF16>(wd[e]);
          s = fmaf(qs[8 * c + 2 * e], f.x, s);
          s = fmaf(qs[8 * c + 2 * e + 1], f.y, s);
        }
      }
      const int kv = k_lo + j;
      x = s;
      if constexpr (MOD == MOD_ALIBI) x = fmaf(slope2, float(kv), x);   // q_idx = 0
      if constexpr (MOD == MOD_CHECKER) x += (kv & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;
      if constexpr (MOD == MOD_CAUSAL) if (kv > 0) x = -INFINITY;
      if (p.key_mask && p.key_mask[(size_t)b * p.Skv + kv] == 0) x = -INFINITY;
    }
  }
  // ---- max over the 128 scores, exponentials, their sum
  float M = x;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  if (lane == 0) redm[warp] = M;
  __syncthreads();
  M = fmaxf(fmaxf(redm[0], redm[1]), fmaxf(redm[2], redm[3]));
  const float Mu = (M == -INFINITY) ? 0.f : M;
  const float pj = ex2(x - Mu);
  sc_s[tid] = pj;
  float ls = pj;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, off);
  if (lane == 0) reds[warp] = ls;
  __syncthreads();
  // ---- o[d] = sum_j p_j v_jd: thread d over keys [0, 64), thread d + 64 over [64, 128)
  {
    const int d = tid & 63, part = tid >> 6;
    float acc = 0.f;
    const int j0 = part * 64, j1 = min(nk, j0 + 64);
    for (int j = j0; j < j1; ++j) {
      const uint16_t raw = vs[j * 64 + d];
      float vf;
      if constexpr (BF16)
        vf = __uint_as_float(static_cast<uint32_t>(raw) << 16);
      else
        asm("cvt.f32.f16 %0, %1;" : "=f"(vf) : "h"(raw));
      acc = fmaf(sc_s[j], vf, acc);
    }
    if (part == 1) o_part[d] = acc;
    __syncthreads();
    float* mine = p.partial + ((size_t)bh * p.nsplit + split) * (2 + 64);
    if (part == 0) {
      mine[2 + d] = acc + o_part[d];
      if (d == 0) {
        mine[0] = M;
        mine[1] = (reds[0] + reds[1]) + (reds[2] + reds[3]);
      }
    }
  }
  if (!ok && tid == 0 && p.status) atomicCAS(p.status, 0, kStatusTimeout | (41 << 8));
  // ---- the last CTA of this (b, h) merges all splits
  __threadfence();
  __syncthreads();
  if (tid == 0) ticket = atomicAdd(p.counter + bh, 1u);
  __syncthreads();
  if (ticket != (unsigned)(p.nsplit - 1)) return;
  __threadfence();
  if (tid < 64) {
    const float* all = p.partial + (size_t)bh * p.nsplit * (2 + 64);
    float Mx = -INFINITY;
    for (int s = 0; s < p.nsplit; ++s) Mx = fmaxf(Mx, __ldcg(all + s * 66));
    const float Mxu = (Mx == -INFINITY) ? 0.f : Mx;
    float Lsum = 0.f, acc = 0.f;
    for (int s = 0; s < p.nsplit; ++s) {
      const float w = ex2(__ldcg(all + s * 66) - Mxu);
      Lsum = fmaf(__ldcg(all + s * 66 + 1), w, Lsum);
      acc = fmaf(__ldcg(all + s * 66 + 2 + tid), w, acc);
    }
    const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
    const float val = acc * inv;
    const float nb = __shfl_down_sync(0xffffffffu, val, 1);
    if ((tid & 1) == 0) {
      uint32_t* op = reinterpret_cast<uint32_t*>(reinterpret_cast<uint16_t*>(p.out) + (size_t)bh * 64 + tid);
      *op = pack2<BF16>(val, nb);
    }
    if (tid == 0) {
      p.lse[bh] = Lsum > 0.f ? (Mxu + lg2(Lsum)) * kLn2 : -INFINITY;
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
  if (p.keys_per_split > DEC_KEYS || p.keys_per_split < 1) return cudaErrorInvalidValue;
  return bf16 ? launch_decode_t<true>(p, st) : launch_decode_t<false>(p, st);
}

}  // namespace attn
