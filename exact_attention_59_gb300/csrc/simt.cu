// simt.cu - the float32 attention path on the FP32 FMA pipe.
//
// f32 inputs are a correctness path (a 256-token case): a tcgen05 kind::tf32
// contraction rounds operands to 10 mantissa bits, which alone exceeds a 1e-4
// output bound, so float32 runs on plain FMA, one thread per query row (or per
// key row in the dK/dV pass), with K/V or Q/dO tiles staged in shared memory.
// The arithmetic is the same online softmax (attnax Pallas kernel body) in
// base 2, with the same tile skipping and masks as the tensor-core kernels.
#include "kernels.h"

namespace attn {

constexpr int SIMT_D = 64;
constexpr int SIMT_CHUNK = 32;
constexpr int SIMT_PAD = SIMT_D + 1;   // conflict-free per-thread row reads

// Per-(q tile, kv block) decision shared by the three kernels.
DEVI uint8_t simt_tile_flags(const SimtParams& p, int b, int h, int qt, int kb, bool all_padded) {
  if (all_padded) return 0;
  const int st = p.bm_tiles ? p.bm_tiles[b * p.bm_sb + h * p.bm_sh + (long long)qt * p.nkb + kb] : TILE_FULL;
  if (st == TILE_EMPTY) return 0;
  return KB_VISIT | ((st == TILE_PARTIAL && p.bm_mod != MASKMOD_NONE) ? KB_MASKMOD : 0);
}

// score in log2 units after scale, score_mod and masks; -inf where masked
DEVI float simt_logit(const SimtParams& p, float dot_sc, int h, int qi, int kj, uint8_t flags, uint8_t key_keep,
                      float slope2) {
  float x = dot_sc;
  if (p.mod == MOD_ALIBI) x = fmaf(slope2, float(kj - qi), x);
  if (p.mod == MOD_CHECKER) x += ((qi + kj) & 1) ? -0.5f * kLog2e : 0.5f * kLog2e;
  const bool causal = p.mod == MOD_CAUSAL || ((flags & KB_MASKMOD) && p.bm_mod == MASKMOD_CAUSAL);
  if (causal && kj > qi) x = -INFINITY;
  if (!key_keep) x = -INFINITY;
  return x;
}

__global__ void __launch_bounds__(128) simt_fwd_kernel(const SimtParams p) {
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;
  const int qi = qt * 128 + threadIdx.x;
  __shared__ float ks[SIMT_CHUNK][SIMT_D], vs[SIMT_CHUNK][SIMT_D];
  __shared__ uint8_t kk[128];
  float q[SIMT_D], o[SIMT_D];
  const float* qrow = p.q + ((size_t)bh * p.Sq + qi) * SIMT_D;
#pragma unroll
  for (int d = 0; d < SIMT_D; ++d) {
    q[d] = qrow[d] * p.sc;
    o[d] = 0.f;
  }
  const float slope2 = alibi_slope_log2(h, p.H);
  float m = -INFINITY, l = 0.f;
  for (int kb = 0; kb < p.nkb; ++kb) {
    const int kv0 = kb * 128;
    const uint8_t keep_t = p.key_mask ? (p.key_mask[(size_t)b * p.Skv + kv0 + threadIdx.x] != 0) : 1;
    kk[threadIdx.x] = keep_t;
    const bool any_keep = __syncthreads_or(keep_t);
    const uint8_t f = simt_tile_flags(p, b, h, qt, kb, !any_keep);
    if (p.visited && threadIdx.x == 0) p.visited[((size_t)bh * p.nqb + qt) * p.nkb + kb] = (f & KB_VISIT) ? 1 : 0;
    if (!(f & KB_VISIT)) continue;
    for (int c0 = 0; c0 < 128; c0 += SIMT_CHUNK) {
      __syncthreads();
      for (int e = threadIdx.x; e < SIMT_CHUNK * SIMT_D; e += 128) {
        const size_t g = ((size_t)bh * p.Skv + kv0 + c0) * SIMT_D + e;
        ks[e / SIMT_D][e % SIMT_D] = p.k[g];
        vs[e / SIMT_D][e % SIMT_D] = p.v[g];
      }
      __syncthreads();
      for (int j = 0; j < SIMT_CHUNK; ++j) {
        float dot = 0.f;
#pragma unroll
        for (int d = 0; d < SIMT_D; ++d) dot = fmaf(q[d], ks[j][d], dot);
        const float x = simt_logit(p, dot, h, qi, kv0 + c0 + j, f, kk[c0 + j], slope2);
        const float m_new = fmaxf(m, x);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = exp2f(m - m_use);
        const float pj = exp2f(x - m_use);
#pragma unroll
        for (int d = 0; d < SIMT_D; ++d) o[d] = fmaf(pj, vs[j][d], o[d] * alpha);
        l = fmaf(l, alpha, pj);
        m = m_new;
      }
    }
    __syncthreads();
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  float* orow = p.o + ((size_t)bh * p.Sq + qi) * SIMT_D;
#pragma unroll
  for (int d = 0; d < SIMT_D; ++d) orow[d] = o[d] * inv;
  const float m_fin = (m == -INFINITY) ? 0.f : m;
  p.lse[(size_t)bh * p.Sq + qi] = l > 0.f ? (m_fin + log2f(l)) * kLn2 : -INFINITY;
}

// One thread per key row; loops over the q rows of every visited q block.
__global__ void __launch_bounds__(128) simt_bwd_dkdv_kernel(const SimtParams p) {
  const int kb = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;
  const int kj = kb * 128 + threadIdx.x;
  extern __shared__ float simt_dyn[];
  float (*krow)[SIMT_PAD] = reinterpret_cast<float (*)[SIMT_PAD]>(simt_dyn);
  float (*vrow)[SIMT_PAD] = reinterpret_cast<float (*)[SIMT_PAD]>(simt_dyn + 128 * SIMT_PAD);
  __shared__ float qs[SIMT_CHUNK][SIMT_D], dos[SIMT_CHUNK][SIMT_D], ls[SIMT_CHUNK], ds_[SIMT_CHUNK];
  for (int e = threadIdx.x; e < 128 * SIMT_D; e += 128) {
    const size_t g = ((size_t)bh * p.Skv + kb * 128) * SIMT_D + e;
    krow[e / SIMT_D][e % SIMT_D] = p.k[g];
    vrow[e / SIMT_D][e % SIMT_D] = p.v[g];
  }
  const uint8_t keep = p.key_mask ? (p.key_mask[(size_t)b * p.Skv + kj] != 0) : 1;
  const bool any_keep = __syncthreads_or(keep);
  const float slope2 = alibi_slope_log2(h, p.H);
  float dk[SIMT_D], dv[SIMT_D];
#pragma unroll
  for (int d = 0; d < SIMT_D; ++d) dk[d] = dv[d] = 0.f;
  for (int qt = 0; qt < p.nqb; ++qt) {
    const uint8_t f = simt_tile_flags(p, b, h, qt, kb, !any_keep);
    if (!(f & KB_VISIT)) continue;
    for (int c0 = 0; c0 < 128; c0 += SIMT_CHUNK) {
      __syncthreads();
      const size_t row0 = (size_t)bh * p.Sq + qt * 128 + c0;
      for (int e = threadIdx.x; e < SIMT_CHUNK * SIMT_D; e += 128) {
        qs[e / SIMT_D][e % SIMT_D] = p.q[row0 * SIMT_D + e];
        dos[e / SIMT_D][e % SIMT_D] = p.dout[row0 * SIMT_D + e];
      }
      if (threadIdx.x < SIMT_CHUNK) {
        ls[threadIdx.x] = p.lse2[row0 + threadIdx.x];
        ds_[threadIdx.x] = p.delta[row0 + threadIdx.x];
      }
      __syncthreads();
      for (int i = 0; i < SIMT_CHUNK; ++i) {
        const int qi = qt * 128 + c0 + i;
        float dot = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < SIMT_D; ++d) {
          dot = fmaf(qs[i][d], krow[threadIdx.x][d], dot);
          dp = fmaf(dos[i][d], vrow[threadIdx.x][d], dp);
        }
        const float x = simt_logit(p, dot * p.sc, h, qi, kj, f, keep, slope2);
        const float pij = exp2f(x + ls[i]);
        const float dsij = pij * (dp + ds_[i]);
#pragma unroll
        for (int d = 0; d < SIMT_D; ++d) {
          dv[d] = fmaf(pij, dos[i][d], dv[d]);
          dk[d] = fmaf(dsij, qs[i][d], dk[d]);
        }
      }
    }
  }
  float* dkr = p.dk + ((size_t)bh * p.Skv + kj) * SIMT_D;
  float* dvr = p.dv + ((size_t)bh * p.Skv + kj) * SIMT_D;
#pragma unroll
  for (int d = 0; d < SIMT_D; ++d) {
    dkr[d] = dk[d] * p.scale;
    dvr[d] = dv[d];
  }
}

// One thread per query row; loops over the keys of every visited kv block.
__global__ void __launch_bounds__(128) simt_bwd_dq_kernel(const SimtParams p) {
  const int qt = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int bh = b * p.H + h;
  const int qi = qt * 128 + threadIdx.x;
  extern __shared__ float simt_dyn[];
  float (*qrow)[SIMT_PAD] = reinterpret_cast<float (*)[SIMT_PAD]>(simt_dyn);
  float (*dorow)[SIMT_PAD] = reinterpret_cast<float (*)[SIMT_PAD]>(simt_dyn + 128 * SIMT_PAD);
  __shared__ float ks[SIMT_CHUNK][SIMT_D], vs[SIMT_CHUNK][SIMT_D];
  __shared__ uint8_t kk[128];
  for (int e = threadIdx.x; e < 128 * SIMT_D; e += 128) {
    const size_t g = ((size_t)bh * p.Sq + qt * 128) * SIMT_D + e;
    qrow[e / SIMT_D][e % SIMT_D] = p.q[g];
    dorow[e / SIMT_D][e % SIMT_D] = p.dout[g];
  }
  const float l2 = p.lse2[(size_t)bh * p.Sq + qi];
  const float dl = p.delta[(size_t)bh * p.Sq + qi];
  const float slope2 = alibi_slope_log2(h, p.H);
  float dq[SIMT_D];
#pragma unroll
  for (int d = 0; d < SIMT_D; ++d) dq[d] = 0.f;
  for (int kb = 0; kb < p.nkb; ++kb) {
    const int kv0 = kb * 128;
    const uint8_t keep_t = p.key_mask ? (p.key_mask[(size_t)b * p.Skv + kv0 + threadIdx.x] != 0) : 1;
    __syncthreads();
    kk[threadIdx.x] = keep_t;
    const bool any_keep = __syncthreads_or(keep_t);
    const uint8_t f = simt_tile_flags(p, b, h, qt, kb, !any_keep);
    if (!(f & KB_VISIT)) continue;
    for (int c0 = 0; c0 < 128; c0 += SIMT_CHUNK) {
      __syncthreads();
      for (int e = threadIdx.x; e < SIMT_CHUNK * SIMT_D; e += 128) {
        const size_t g = ((size_t)bh * p.Skv + kv0 + c0) * SIMT_D + e;
        ks[e / SIMT_D][e % SIMT_D] = p.k[g];
        vs[e / SIMT_D][e % SIMT_D] = p.v[g];
      }
      __syncthreads();
      for (int j = 0; j < SIMT_CHUNK; ++j) {
        float dot = 0.f, dp = 0.f;
#pragma unroll
        for (int d = 0; d < SIMT_D; ++d) {
          dot = fmaf(qrow[threadIdx.x][d], ks[j][d], dot);
          dp = fmaf(dorow[threadIdx.x][d], vs[j][d], dp);
        }
        const float x = simt_logit(p, dot * p.sc, h, qi, kv0 + c0 + j, f, kk[c0 + j], slope2);
        const float pij = exp2f(x + l2);
        const float dsij = pij * (dp + dl);
#pragma unroll
        for (int d = 0; d < SIMT_D; ++d) dq[d] = fmaf(dsij, ks[j][d], dq[d]);
      }
    }
  }
  float* out = p.dq + ((size_t)bh * p.Sq + qi) * SIMT_D;
#pragma unroll
  for (int d = 0; d < SIMT_D; ++d) out[d] = dq[d] * p.scale;
}

cudaError_t launch_simt_fwd(const SimtParams& p, cudaStream_t st) {
  simt_fwd_kernel<<<dim3(p.nqb, p.H, p.B), 128, 0, st>>>(p);
  return cudaGetLastError();
}
constexpr int SIMT_DYN_BYTES = 2 * 128 * SIMT_PAD * 4;

cudaError_t launch_simt_bwd_dkdv(const SimtParams& p, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(simt_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SIMT_DYN_BYTES);
  if (e != cudaSuccess) return e;
  simt_bwd_dkdv_kernel<<<dim3(p.nkb, p.H, p.B), 128, SIMT_DYN_BYTES, st>>>(p);
  return cudaGetLastError();
}
cudaError_t launch_simt_bwd_dq(const SimtParams& p, cudaStream_t st) {
  cudaError_t e = cudaFuncSetAttribute(simt_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SIMT_DYN_BYTES);
  if (e != cudaSuccess) return e;
  simt_bwd_dq_kernel<<<dim3(p.nqb, p.H, p.B), 128, SIMT_DYN_BYTES, st>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
