// decode_noalloc.cu - single-query decode for callers that cannot allocate.
//
// attn_decode() needs a caller-provided workspace for its split-KV partial
// results and its completion tickets.  Some callers have no way to provide
// one: a plugin or operator running inside a host framework that owns all
// device memory and exposes no allocation hook, or a latency-critical serving
// loop whose device memory plan is frozen at start-up and that must not call
// cudaMalloc (or a caching allocator that may call it) while serving.  For
// them, attn_decode_noalloc() keeps that scratch in a fixed array compiled
// into this library instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kDecodeScratchBytes of it until the process exits.  Host code
// cannot use the array's name as a device address, so each call looks the
// address up with cudaGetSymbolAddress on the current device.  The first call
// on a device also loads this library's device code there (set-up work that
// belongs before any stream capture); later look-ups are cheap, and a fresh
// look-up stays right after cudaDeviceReset or under another context, where a
// remembered address would point at memory that is no longer mapped.
#include <cmath>

#include "../../include/attn.h"
#include "kernels.h"

namespace {

constexpr size_t kDecodeScratchBytes = size_t(4) << 20;   // 4 MiB per device

static __device__ __align__(256) unsigned char g_decode_scratch[kDecodeScratchBytes];

// Device address of the built-in scratch on the current device.
attn_status scratch_address(void** addr) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return ATTN_ERR_CUDA;
  }
  *addr = p;
  return ATTN_OK;
}

bool is_aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" attn_status attn_decode_noalloc(const attn_shape* s, const void* q, const void* k, const void* v,
                                           const uint8_t* key_mask, attn_score_mod mod, float scale, void* out,
                                           float* lse, attn_stream_t stream) {
  using namespace attn;
  if (!s || s->B <= 0 || s->H <= 0 || s->Sq <= 0 || s->Skv <= 0 || s->D <= 0) return ATTN_ERR_INVALID_ARG;
  if (s->dtype != ATTN_F16 && s->dtype != ATTN_BF16 && s->dtype != ATTN_F32) return ATTN_ERR_INVALID_ARG;
  if (s->Sq != 1) return ATTN_ERR_SHAPE;
  if (s->D != 64 || s->dtype == ATTN_F32) return ATTN_ERR_UNSUPPORTED;
  if ((int)mod < 0 || (int)mod > 3 || !std::isfinite(scale) || scale == 0.f)
    return ATTN_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || !lse) return ATTN_ERR_INVALID_ARG;
  if (!is_aligned16(q) || !is_aligned16(k) || !is_aligned16(v) || !is_aligned16(out) || !is_aligned16(lse) ||
      (key_mask && !is_aligned16(key_mask)))
    return ATTN_ERR_ALIGN;
  if ((long long)s->B * s->H * s->Skv > (1LL << 31) - 1) return ATTN_ERR_SHAPE;

  // Same split of the keys as attn_decode, so both entry points give the same result.
  const long long BH = (long long)s->B * s->H;
  int nsplit = decode_num_splits(s->B, s->H, s->Skv);
  const int kps = (s->Skv + nsplit - 1) / nsplit;
  nsplit = (s->Skv + kps - 1) / kps;
  const size_t partial_bytes = align256((size_t)BH * nsplit * (2 + 64) * sizeof(float));
  const size_t counter_bytes = (size_t)BH * sizeof(unsigned);
  if (partial_bytes + counter_bytes > kDecodeScratchBytes) return ATTN_ERR_WORKSPACE;   // shape too large

  void* base = nullptr;
  const attn_status st = scratch_address(&base);
  if (st != ATTN_OK) return st;
  float* partial = static_cast<float*>(base);
  unsigned* counter = reinterpret_cast<unsigned*>(static_cast<unsigned char*>(base) + partial_bytes);

  DecodeParams p{};
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.lse = lse;
  p.key_mask = key_mask;
  p.partial = partial;
  p.counter = counter;
  p.B = s->B;
  p.H = s->H;
  p.Skv = s->Skv;
  p.nsplit = nsplit;
  p.keys_per_split = kps;
  p.sc = scale * kLog2e;
  p.mod = (int)mod;
  return launch_decode(p, s->dtype == ATTN_BF16, (cudaStream_t)stream) == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
