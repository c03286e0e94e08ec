// api.cu - the C ABI declared in include/attn.h: validation, workspace
// layout, TMA descriptor encoding and kernel dispatch.  No allocation, no
// synchronisation (except attn_poll_status), no state beyond one cached
// process-wide value (the CUDA driver's tensor-map encoder).
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/attn.h"
#include "kernels.h"
#include "usermod.h"

using namespace attn;

// Device-side wait limit, read at every call (ATTN_TIMEOUT_NS, default 2 s).
unsigned long long attn::attn_timeout_ns() {
  const char* e = std::getenv("ATTN_TIMEOUT_NS");
  unsigned long long v = 2000000000ULL;
  if (e && *e) {
    char* end = nullptr;
    const unsigned long long x = std::strtoull(e, &end, 10);
    if (end && *end == '\0' && x > 0) v = x;
  }
  return v;
}

namespace {

constexpr long long kMaxRows = (1LL << 31) - 1;

unsigned long long timeout_ns() { return attn::attn_timeout_ns(); }

// Test hook, off unless ATTN_DEBUG_INJECT_STALL=1: the D = 64 forward's producer
// withholds its first K/V copy, so the kernel's bounded waits run out and it
// reports ATTN_ERR_TIMEOUT through the status word (no trap, no fault).
int inject_stall() {
  const char* e = std::getenv("ATTN_DEBUG_INJECT_STALL");
  return (e && e[0] == '1' && e[1] == '\0') ? 1 : 0;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D view (rows, cols) of a row-major tensor, box {64 columns, 128 rows}, 128-byte swizzle.
bool make_tmap(CUtensorMap* m, const void* base, long long rows, int cols, attn_dtype dt) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  const CUtensorMapDataType t = dt == ATTN_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, t, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
size_t esize(attn_dtype d) { return d == ATTN_F32 ? 4 : 2; }

bool shape_ok(const attn_shape* s) {
  return s && s->B > 0 && s->H > 0 && s->Sq > 0 && s->Skv > 0 && s->D > 0 &&
         (s->dtype == ATTN_F32 || s->dtype == ATTN_F16 || s->dtype == ATTN_BF16) &&
         (long long)s->B * s->H * s->Sq <= kMaxRows && (long long)s->B * s->H * s->Skv <= kMaxRows;
}

struct DecodeSplit {
  int nsplit, kps;
};
DecodeSplit decode_split(const attn_shape* s) {
  int ns = decode_num_splits(s->B, s->H, s->Skv);
  const int kps = (s->Skv + ns - 1) / ns;
  ns = (s->Skv + kps - 1) / kps;
  return {ns, kps};
}

// 128-row tiles covering n rows (the last one may be partial)
int tiles_of(int n) { return (n + 127) / 128; }

// Streaming multiprocessors of the current device (152 on a GB300; the same
// number is assumed when no device can be queried, e.g. for a size query on a
// machine without a GPU).
long long sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      n <= 0) {
    (void)cudaGetLastError();   // leave no stale error for a later launch check
    return 152;
  }
  return n;
}

// Split of a query chunk's kv blocks over CTAs: about one CTA per SM in total
// (the forward kernel runs one CTA per SM), at least one kv block each.
struct ChunkSplit {
  int nsplit, kps;
};
ChunkSplit chunk_split(const attn_shape* s) {
  const long long nkb = tiles_of(s->Skv), items = (long long)s->B * s->H * ((tiles_of(s->Sq) + 1) / 2);
  int ns = (int)std::max<long long>(1, std::min<long long>(nkb, sm_count() / std::max<long long>(1, items)));
  const int kps = (int)((nkb + ns - 1) / ns);
  ns = (int)((nkb + kps - 1) / kps);
  return {ns, kps};
}

WsLayout layout(attn_op op, const attn_shape* s) {
  WsLayout w;
  size_t off = 256;
  const size_t B = s->B, BH = (size_t)s->B * s->H;
  w.km_bits = off;
  off = align256(off + B * ((s->Skv + 31) / 32) * 4);
  w.km_sum = off;
  off = align256(off + B * ((s->Skv + 127) / 128));
  if (op == ATTN_OP_BWD) {
    w.delta = off;
    off = align256(off + BH * s->Sq * 4);
    w.lse2 = off;
    off = align256(off + BH * s->Sq * 4);
  }
  if (op == ATTN_OP_DECODE) {
    const DecodeSplit d = decode_split(s);
    w.partial = off;
    off = align256(off + BH * d.nsplit * (2 + 64) * 4);
    w.counter = off;
    off = align256(off + BH * 4);
  }
  if (op == ATTN_OP_DECODE_CHUNK) {
    // partial rows of the split: sized for min(max(items, SMs), items * nkb) CTAs,
    // a bound on items * nsplit that grows with every dimension of the shape
    const long long items = (long long)BH * ((tiles_of(s->Sq) + 1) / 2), nkb = tiles_of(s->Skv);
    const long long ctas = std::min(std::max(items, sm_count()), items * nkb);
    w.partial = off;
    off = align256(off + (size_t)ctas * 256 * FWD_PART * 4);
  }
  w.total = off;
  return w;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<uint8_t*>(ws) + off);
}

attn_status cuda_status(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

// Checks shared by every prefill call.  Any Sq, Skv >= 1 on the f16/bf16
// D = 64 path (the last q and kv tiles may be partial); multiples of 128 for
// f32 and D = 512.
attn_status check_prefill(const attn_shape* s, bool backward) {
  if (!shape_ok(s)) return ATTN_ERR_INVALID_ARG;
  const bool ragged_ok = s->D == 64;
  if (!ragged_ok && (s->Sq % 128 != 0 || s->Skv % 128 != 0)) return ATTN_ERR_SHAPE;
  if (tiles_of(s->Skv) > FWD_MAXKB || tiles_of(s->Sq) > FWD_MAXKB) return ATTN_ERR_SHAPE;
  (void)backward;   // D = 512 has a forward and a backward, f16/bf16
  if (s->D == 64) return ATTN_OK;
  if (s->D == 512 && s->dtype != ATTN_F32) return ATTN_OK;
  return ATTN_ERR_UNSUPPORTED;
}

// Whether the ALiBi / checkerboard bias rides on the score products (three 16-bit
// terms of bias / scale in one more K = 16 MMA step): needs scale != 0 and a
// term of at most 2^12, where the f32 sum of S and the term keeps S to about
// 2^-11 of its scale-free units (1/sqrt(D) scales give 4 for the checkerboard
// and 2^(-8/H) 127 / scale <= 1016 for ALiBi at D <= 64).  Otherwise the
// kernels add the bias per score.
int mod_fold_ok(attn_score_mod mod, float scale, int H) {
  if (scale == 0.f || !std::isfinite(scale)) return 0;
  const float inv = 1.f / std::fabs(scale);
  if (mod == ATTN_MOD_CHECKERBOARD) return 0.5f * inv <= 4096.f ? 1 : 0;
  if (mod == ATTN_MOD_ALIBI) return std::exp2(-8.0f / float(H)) * 127.f * inv <= 4096.f ? 1 : 0;
  return 0;
}

// The scale must be finite and nonzero: the D = 64 kernels carry masks and the
// dK/dV pass's -lse / scale as terms of their score products, which the scale
// multiplies afterwards (the pages' scale is 1/sqrt(D), never 0).
attn_status check_mod(attn_score_mod mod, float scale) {
  if ((int)mod < 0 || (int)mod > 3) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale == 0.f) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// A block mask; mask_mod ATTN_MASKMOD_USER only with a user mod that has a mask
// expression (`user_mask`).
attn_status check_bm(const attn_block_mask* bm, bool user_mask = false) {
  if (!bm) return ATTN_OK;
  if (!bm->tiles) return ATTN_ERR_INVALID_ARG;
  if ((int)bm->mask_mod < 0 || (int)bm->mask_mod > (user_mask ? 2 : 1)) return ATTN_ERR_INVALID_ARG;
  if (bm->block_q != 128 || bm->block_kv != 128) return ATTN_ERR_UNSUPPORTED;
  return ATTN_OK;
}

attn_status check_ws(attn_op op, const attn_shape* s, void* ws, size_t ws_bytes) {
  if (!ws) return ATTN_ERR_WORKSPACE;
  if (!aligned(ws, 256)) return ATTN_ERR_ALIGN;
  if (ws_bytes < layout(op, s).total) return ATTN_ERR_WORKSPACE;
  return ATTN_OK;
}

void bm_strides(const attn_shape* s, const attn_block_mask* bm, long long& sb, long long& sh) {
  const long long tile = (long long)tiles_of(s->Sq) * tiles_of(s->Skv);
  sh = bm->bcast_h ? 0 : tile;
  sb = bm->bcast_b ? 0 : (bm->bcast_h ? 1 : s->H) * tile;
}

#define ATTN_TRY(x)                   \
  do {                                \
    const attn_status _st = (x);      \
    if (_st != ATTN_OK) return _st;   \
  } while (0)

#define ATTN_PTR(p)                                  \
  do {                                               \
    if (!(p)) return ATTN_ERR_INVALID_ARG;           \
    if (!aligned((p), 16)) return ATTN_ERR_ALIGN;    \
  } while (0)

#define ATTN_OPT_PTR(p)                              \
  do {                                               \
    if ((p) && !aligned((p), 16)) return ATTN_ERR_ALIGN; \
  } while (0)

attn_status run_keymask(const attn_shape* s, const uint8_t* km, void* ws, cudaStream_t st) {
  if (!km) return ATTN_OK;
  const WsLayout w = layout(ATTN_OP_FWD, s);
  return cuda_status(launch_keymask_pack(km, s->B, s->Skv, at<uint32_t>(ws, w.km_bits), at<uint8_t>(ws, w.km_sum), st));
}

BwdParams bwd_params(const attn_shape* s, const void* q, const void* k, const void* v, const void* dout,
                     const uint8_t* key_mask, const attn_block_mask* bm, attn_score_mod mod, float scale, void* ws,
                     bool& ok) {
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  const long long rq = (long long)s->B * s->H * s->Sq, rk = (long long)s->B * s->H * s->Skv;
  ok = true;
  if (s->dtype != ATTN_F32) {
    ok = make_tmap(&p.tm_q, q, rq, s->D, s->dtype) && make_tmap(&p.tm_k, k, rk, s->D, s->dtype) &&
         make_tmap(&p.tm_v, v, rk, s->D, s->dtype) && make_tmap(&p.tm_do, dout, rq, s->D, s->dtype);
  }
  const WsLayout wb = layout(ATTN_OP_BWD, s);
  p.delta = at<float>(ws, wb.delta);
  p.lse2 = at<float>(ws, wb.lse2);
  p.km_bits = key_mask ? at<uint32_t>(ws, wb.km_bits) : nullptr;
  p.km_sum = key_mask ? at<uint8_t>(ws, wb.km_sum) : nullptr;
  p.bm_tiles = bm ? bm->tiles : nullptr;
  if (bm) bm_strides(s, bm, p.bm_sb, p.bm_sh);
  p.bm_mod = bm ? (int)bm->mask_mod : 0;
  p.status = at<int>(ws, 0);
  p.B = s->B;
  p.H = s->H;
  p.Sq = s->Sq;
  p.Skv = s->Skv;
  p.nqb = tiles_of(s->Sq);
  p.nkb = tiles_of(s->Skv);
  p.sc = scale * kLog2e;
  p.scale = scale;
  p.timeout_ns = timeout_ns();
  p.fold = mod_fold_ok(mod, scale, s->H);
  p.inv_scale = scale != 0.f ? 1.f / scale : 0.f;
  return p;
}

SimtParams simt_params(const attn_shape* s, const void* q, const void* k, const void* v, const uint8_t* key_mask,
                       const attn_block_mask* bm, attn_score_mod mod, float scale) {
  SimtParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = (const float*)q;
  p.k = (const float*)k;
  p.v = (const float*)v;
  p.key_mask = key_mask;
  p.bm_tiles = bm ? bm->tiles : nullptr;
  if (bm) bm_strides(s, bm, p.bm_sb, p.bm_sh);
  p.bm_mod = bm ? (int)bm->mask_mod : 0;
  p.B = s->B;
  p.H = s->H;
  p.Sq = s->Sq;
  p.Skv = s->Skv;
  p.nqb = tiles_of(s->Sq);
  p.nkb = tiles_of(s->Skv);
  p.mod = (int)mod;
  p.sc = scale * kLog2e;
  p.scale = scale;
  p.timeout_ns = timeout_ns();
  return p;
}

long long dense_mask_count(const attn_shape* s, int bcast_b, int bcast_h) {
  return (long long)(bcast_b ? 1 : s->B) * (bcast_h ? 1 : s->H);
}

// A dense mask rides on the f16/bf16 D = 64 path only.
attn_status check_dm(const attn_shape* s, const attn_dense_mask* dm) {
  if (!dm) return ATTN_OK;
  if (!dm->packed || (dm->bcast_b != 0 && dm->bcast_b != 1) || (dm->bcast_h != 0 && dm->bcast_h != 1))
    return ATTN_ERR_INVALID_ARG;
  if (!aligned(dm->packed, 256)) return ATTN_ERR_ALIGN;
  if (s->D != 64) return ATTN_ERR_UNSUPPORTED;
  if (dm->packed_bytes < dense_mask_layout(dense_mask_count(s, dm->bcast_b, dm->bcast_h), s->Sq, s->Skv).total)
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

DenseMaskView dm_view(const attn_shape* s, const attn_dense_mask* dm) {
  DenseMaskView v;
  std::memset(&v, 0, sizeof(v));
  if (!dm) return v;
  const DenseMaskLayout l = dense_mask_layout(dense_mask_count(s, dm->bcast_b, dm->bcast_h), s->Sq, s->Skv);
  const uint8_t* base = static_cast<const uint8_t*>(dm->packed);
  v.tiles = base + l.tiles;
  v.rowbits = reinterpret_cast<const uint32_t*>(base + l.rowbits);
  v.colbits = reinterpret_cast<const uint32_t*>(base + l.colbits);
  v.mh = dm->bcast_h ? 0 : 1;
  v.mb = dm->bcast_b ? 0 : (dm->bcast_h ? 1 : s->H);
  return v;
}

}  // namespace

extern "C" {

size_t attn_workspace_size(attn_op op, const attn_shape* shape) {
  if (!shape_ok(shape)) return 0;
  if ((int)op < 0 || (int)op > 3) return 0;
  return layout(op, shape).total;
}

const char* attn_status_string(attn_status s) {
  switch (s) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_SHAPE: return "unsupported shape (f32 and D=512 prefill need Sq, Skv multiples of 128; decode needs Sq == 1)";
    case ATTN_ERR_ALIGN: return "pointer not 16-byte aligned (workspace: 256-byte)";
    case ATTN_ERR_UNSUPPORTED: return "dtype / head dim / mod / block size combination not built";
    case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
    case ATTN_ERR_CUDA: return "CUDA error";
    case ATTN_ERR_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

attn_status attn_build_block_mask(attn_mask_mod mask_mod, int B, int H, int Sq, int Skv, int bq, int bkv,
                                  uint8_t* tiles, attn_stream_t stream) {
  if (B <= 0 || H <= 0 || Sq <= 0 || Skv <= 0 || bq <= 0 || bkv <= 0 || !tiles) return ATTN_ERR_INVALID_ARG;
  if ((int)mask_mod < 0 || (int)mask_mod > 1) return ATTN_ERR_INVALID_ARG;
  return cuda_status(launch_build_block_mask((int)mask_mod, B, H, Sq, Skv, bq, bkv, tiles, (cudaStream_t)stream));
}

attn_status attn_fwd(const attn_shape* s, const void* q, const void* k, const void* v, const uint8_t* key_mask,
                     const attn_block_mask* bm, attn_score_mod mod, float scale, void* out, float* lse, void* ws,
                     size_t ws_bytes, attn_stream_t stream, uint8_t* debug_visited) {
  return attn_fwd_dense(s, q, k, v, key_mask, nullptr, bm, mod, scale, out, lse, ws, ws_bytes, stream, debug_visited);
}

// The forward behind attn_fwd, attn_fwd_dense and attn_fwd_user (um: a
// run-time-compiled score_mod in place of `mod`, or NULL).
static attn_status fwd_impl(const attn_shape* s, const void* q, const void* k, const void* v, const uint8_t* key_mask,
                            const attn_dense_mask* dm, const attn_block_mask* bm, attn_score_mod mod, float scale,
                            void* out, float* lse, void* ws, size_t ws_bytes, attn_stream_t stream,
                            uint8_t* debug_visited, attn_user_mod um) {
  ATTN_TRY(check_prefill(s, false));
  ATTN_TRY(check_mod(mod, scale));
  ATTN_TRY(check_bm(bm, um && user_mod_has_mask(um)));
  ATTN_TRY(check_dm(s, dm));
  // the user kernels: D = 64, the 16-bit dtype they were built for, no dense mask
  if (um && (s->D != 64 || s->dtype == ATTN_F32 || dm)) return ATTN_ERR_UNSUPPORTED;
  ATTN_PTR(q);
  ATTN_PTR(k);
  ATTN_PTR(v);
  ATTN_PTR(out);
  ATTN_PTR(lse);
  ATTN_OPT_PTR(key_mask);
  ATTN_TRY(check_ws(ATTN_OP_FWD, s, ws, ws_bytes));
  const void* uk[3] = {nullptr, nullptr, nullptr};
  if (um) ATTN_TRY(user_mod_kernels(um, s->dtype, uk));   // loads the mod's code on this device (first use)
  cudaStream_t st = (cudaStream_t)stream;
  if (s->D == 512) {
    FwdBigParams p;
    std::memset(&p, 0, sizeof(p));
    const long long rq = (long long)s->B * s->H * s->Sq, rk = (long long)s->B * s->H * s->Skv;
    if (!make_tmap(&p.tm_q, q, rq, 512, s->dtype) || !make_tmap(&p.tm_k, k, rk, 512, s->dtype) ||
        !make_tmap(&p.tm_v, v, rk, 512, s->dtype))
      return ATTN_ERR_CUDA;
    ATTN_TRY(run_keymask(s, key_mask, ws, st));
    const WsLayout wl = layout(ATTN_OP_FWD, s);
    p.km_bits = key_mask ? at<uint32_t>(ws, wl.km_bits) : nullptr;
    p.km_sum = key_mask ? at<uint8_t>(ws, wl.km_sum) : nullptr;
    p.out = out;
    p.lse = lse;
    p.bm_tiles = bm ? bm->tiles : nullptr;
    if (bm) bm_strides(s, bm, p.bm_sb, p.bm_sh);
    p.bm_mod = bm ? (int)bm->mask_mod : 0;
    p.visited = debug_visited;
    p.status = at<int>(ws, 0);
    p.B = s->B;
    p.H = s->H;
    p.Sq = s->Sq;
    p.Skv = s->Skv;
    p.nqb = tiles_of(s->Sq);
    p.nkb = tiles_of(s->Skv);
    p.sc = scale * kLog2e;
    p.timeout_ns = timeout_ns();
    return cuda_status(launch_fwd_d512(p, s->dtype == ATTN_BF16, (int)mod, st));
  }
  if (s->dtype == ATTN_F32) {
    SimtParams p = simt_params(s, q, k, v, key_mask, bm, mod, scale);
    p.dm = dm_view(s, dm);
    p.o = (float*)out;
    p.lse = lse;
    p.visited = debug_visited;
    p.status = at<int>(ws, 0);
    return cuda_status(launch_f32_fwd(p, st));
  }
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const long long rq = (long long)s->B * s->H * s->Sq, rk = (long long)s->B * s->H * s->Skv;
  if (!make_tmap(&p.tm_q, q, rq, 64, s->dtype) || !make_tmap(&p.tm_k, k, rk, 64, s->dtype) ||
      !make_tmap(&p.tm_v, v, rk, 64, s->dtype))
    return ATTN_ERR_CUDA;
  p.out = out;
  p.lse = lse;
  p.km = key_mask;   // read as bytes by the kernel's producer: no packing launch
  p.bm_tiles = bm ? bm->tiles : nullptr;
  if (bm) bm_strides(s, bm, p.bm_sb, p.bm_sh);
  p.bm_mod = bm ? (int)bm->mask_mod : 0;
  p.dm = dm_view(s, dm);
  p.visited = debug_visited;
  p.status = at<int>(ws, 0);
  p.B = s->B;
  p.H = s->H;
  p.Sq = s->Sq;
  p.Skv = s->Skv;
  p.nqb = tiles_of(s->Sq);
  p.nkb = tiles_of(s->Skv);
  p.npairs = (p.nqb + 1) / 2;
  p.sc = scale * kLog2e;
  p.timeout_ns = timeout_ns();
  p.inject_stall = inject_stall();
  p.fold = um ? 0 : mod_fold_ok(mod, scale, s->H);
  p.inv_scale = scale != 0.f ? 1.f / scale : 0.f;
  p.nsplit = 1;   // whole kv range per CTA, q_off = 0
  // persistent CTAs, one per SM, taking the items from the counter in the
  // workspace header (kWsItemCounter)
  p.items = at<unsigned>(ws, kWsItemCounter);
  p.ctas = (int)std::min<long long>((long long)p.npairs * p.B * p.H, sm_count());
  {
    // the pairs past the last full round as single tiles, when every pair has two
    // tiles, the split pairs fit one round, and the items are all alike (with a
    // block mask or the causal rule the last items are the shortest: nothing to
    // gain)
    const long long n = (long long)p.npairs * p.B * p.H, rem = n % p.ctas;
    const bool alike = bm == nullptr && mod != ATTN_MOD_CAUSAL;
    p.single_tail = (alike && p.nqb % 2 == 0 && rem > 0 && 2 * rem <= p.ctas) ? 1 : 0;
    p.n_whole = (int)(p.single_tail ? n - rem : n);
  }
  if (um) return cuda_status(launch_fwd_d64_kernel(p, uk[0], st));
  return cuda_status(launch_fwd_d64(p, s->dtype == ATTN_BF16, (int)mod, st));
}

attn_status attn_fwd_dense(const attn_shape* s, const void* q, const void* k, const void* v, const uint8_t* key_mask,
                           const attn_dense_mask* dm, const attn_block_mask* bm, attn_score_mod mod, float scale,
                           void* out, float* lse, void* ws, size_t ws_bytes, attn_stream_t stream,
                           uint8_t* debug_visited) {
  return fwd_impl(s, q, k, v, key_mask, dm, bm, mod, scale, out, lse, ws, ws_bytes, stream, debug_visited, nullptr);
}

attn_status attn_fwd_user(const attn_shape* s, const void* q, const void* k, const void* v, const uint8_t* key_mask,
                          attn_user_mod um, const attn_block_mask* bm, float scale, void* out, float* lse, void* ws,
                          size_t ws_bytes, attn_stream_t stream, uint8_t* debug_visited) {
  if (!um) return ATTN_ERR_INVALID_ARG;
  return fwd_impl(s, q, k, v, key_mask, nullptr, bm, ATTN_MOD_NONE, scale, out, lse, ws, ws_bytes, stream,
                  debug_visited, um);
}

attn_status attn_bwd_preprocess(const attn_shape* s, const void* out, const float* lse, const void* dout,
                                const uint8_t* key_mask, void* ws, size_t ws_bytes, attn_stream_t stream) {
  ATTN_TRY(check_prefill(s, true));
  ATTN_PTR(out);
  ATTN_PTR(lse);
  ATTN_PTR(dout);
  ATTN_OPT_PTR(key_mask);
  ATTN_TRY(check_ws(ATTN_OP_BWD, s, ws, ws_bytes));
  cudaStream_t st = (cudaStream_t)stream;
  const WsLayout w = layout(ATTN_OP_BWD, s);
  // the key mask is packed by the same launch (bits and block summary for the two passes)
  return cuda_status(launch_bwd_preprocess(out, dout, lse, (int)s->dtype, (long long)s->B * s->H * s->Sq, s->D,
                                           at<float>(ws, w.delta), at<float>(ws, w.lse2), key_mask, s->B, s->Skv,
                                           at<uint32_t>(ws, w.km_bits), at<uint8_t>(ws, w.km_sum), st));
}

}  // extern "C"

namespace {

attn_status bwd_dkdv_impl(const attn_shape* s, const void* q, const void* k, const void* v, const void* dout,
                          const uint8_t* key_mask, const attn_dense_mask* dm, const attn_block_mask* bm,
                          attn_score_mod mod, float scale, void* dk, void* dv, void* ws, size_t ws_bytes,
                          attn_stream_t stream, const void* ukern = nullptr, bool user_mask = false) {
  ATTN_TRY(check_prefill(s, true));
  ATTN_TRY(check_dm(s, dm));
  ATTN_TRY(check_mod(mod, scale));
  ATTN_TRY(check_bm(bm, user_mask));
  ATTN_PTR(q);
  ATTN_PTR(k);
  ATTN_PTR(v);
  ATTN_PTR(dout);
  ATTN_PTR(dk);
  ATTN_PTR(dv);
  ATTN_OPT_PTR(key_mask);
  ATTN_TRY(check_ws(ATTN_OP_BWD, s, ws, ws_bytes));
  cudaStream_t st = (cudaStream_t)stream;
  if (s->dtype == ATTN_F32) {
    SimtParams p = simt_params(s, q, k, v, key_mask, bm, mod, scale);
    p.dm = dm_view(s, dm);
    const WsLayout w = layout(ATTN_OP_BWD, s);
    p.dout = (const float*)dout;
    p.dk = (float*)dk;
    p.dv = (float*)dv;
    p.delta = at<float>(ws, w.delta);
    p.lse2 = at<float>(ws, w.lse2);
    p.status = at<int>(ws, 0);
    return cuda_status(launch_f32_dkdv(p, st));
  }
  bool ok;
  BwdParams p = bwd_params(s, q, k, v, dout, key_mask, bm, mod, scale, ws, ok);
  if (!ok) return ATTN_ERR_CUDA;
  p.dk = dk;
  p.dv = dv;
  p.dm = dm_view(s, dm);
  if (s->D == 512) return cuda_status(launch_bwd512_dkdv(p, s->dtype == ATTN_BF16, (int)mod, st));
  // persistent CTAs, one per SM, taking the items from the counter in the
  // workspace header (kWsDkdvCounter)
  p.items = at<unsigned>(ws, kWsDkdvCounter);
  p.ctas = (int)std::min<long long>((long long)p.nkb * p.B * p.H, sm_count());
  if (ukern) return cuda_status(launch_bwd_kernel(p, ukern, true, st));
  return cuda_status(launch_bwd_dkdv(p, s->dtype == ATTN_BF16, (int)mod, st));
}

attn_status bwd_dq_impl(const attn_shape* s, const void* q, const void* k, const void* v, const void* dout,
                        const uint8_t* key_mask, const attn_dense_mask* dm, const attn_block_mask* bm,
                        attn_score_mod mod, float scale, void* dq, void* ws, size_t ws_bytes, attn_stream_t stream,
                        const void* ukern = nullptr, bool user_mask = false) {
  ATTN_TRY(check_prefill(s, true));
  ATTN_TRY(check_dm(s, dm));
  ATTN_TRY(check_mod(mod, scale));
  ATTN_TRY(check_bm(bm, user_mask));
  ATTN_PTR(q);
  ATTN_PTR(k);
  ATTN_PTR(v);
  ATTN_PTR(dout);
  ATTN_PTR(dq);
  ATTN_OPT_PTR(key_mask);
  ATTN_TRY(check_ws(ATTN_OP_BWD, s, ws, ws_bytes));
  cudaStream_t st = (cudaStream_t)stream;
  if (s->dtype == ATTN_F32) {
    SimtParams p = simt_params(s, q, k, v, key_mask, bm, mod, scale);
    p.dm = dm_view(s, dm);
    const WsLayout w = layout(ATTN_OP_BWD, s);
    p.dout = (const float*)dout;
    p.dq = (float*)dq;
    p.delta = at<float>(ws, w.delta);
    p.lse2 = at<float>(ws, w.lse2);
    p.status = at<int>(ws, 0);
    return cuda_status(launch_f32_dq(p, st));
  }
  bool ok;
  BwdParams p = bwd_params(s, q, k, v, dout, key_mask, bm, mod, scale, ws, ok);
  if (!ok) return ATTN_ERR_CUDA;
  p.dq = dq;
  p.dm = dm_view(s, dm);
  if (s->D == 512) return cuda_status(launch_bwd512_dq(p, s->dtype == ATTN_BF16, (int)mod, st));
  // persistent CTAs, one per SM, taking the items from the counter in the
  // workspace header (kWsDqCounter)
  p.items = at<unsigned>(ws, kWsDqCounter);
  p.ctas = (int)std::min<long long>((long long)p.nqb * p.B * p.H, sm_count());
  if (ukern) return cuda_status(launch_bwd_kernel(p, ukern, false, st));
  return cuda_status(launch_bwd_dq(p, s->dtype == ATTN_BF16, (int)mod, st));
}

}  // namespace

extern "C" {

attn_status attn_bwd_dkdv(const attn_shape* s, const void* q, const void* k, const void* v, const void* dout,
                          const uint8_t* key_mask, const attn_block_mask* bm, attn_score_mod mod, float scale,
                          void* dk, void* dv, void* ws, size_t ws_bytes, attn_stream_t stream) {
  return bwd_dkdv_impl(s, q, k, v, dout, key_mask, nullptr, bm, mod, scale, dk, dv, ws, ws_bytes, stream);
}

attn_status attn_bwd_dq(const attn_shape* s, const void* q, const void* k, const void* v, const void* dout,
                        const uint8_t* key_mask, const attn_block_mask* bm, attn_score_mod mod, float scale, void* dq,
                        void* ws, size_t ws_bytes, attn_stream_t stream) {
  return bwd_dq_impl(s, q, k, v, dout, key_mask, nullptr, bm, mod, scale, dq, ws, ws_bytes, stream);
}

attn_status attn_bwd(const attn_shape* s, const void* q, const void* k, const void* v, const void* out,
                     const float* lse, const void* dout, const uint8_t* key_mask, const attn_block_mask* bm,
                     attn_score_mod mod, float scale, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                     attn_stream_t stream) {
  return attn_bwd_dense(s, q, k, v, out, lse, dout, key_mask, nullptr, bm, mod, scale, dq, dk, dv, ws, ws_bytes,
                        stream);
}

// The backward behind attn_bwd, attn_bwd_dense and attn_bwd_user.
static attn_status bwd_all(const attn_shape* s, const void* q, const void* k, const void* v, const void* out,
                           const float* lse, const void* dout, const uint8_t* key_mask, const attn_dense_mask* dm,
                           const attn_block_mask* bm, attn_score_mod mod, float scale, void* dq, void* dk, void* dv,
                           void* ws, size_t ws_bytes, attn_stream_t stream, attn_user_mod um) {
  // validate everything before the first launch
  const bool umask = um && user_mod_has_mask(um);
  ATTN_TRY(check_prefill(s, true));
  ATTN_TRY(check_mod(mod, scale));
  ATTN_TRY(check_bm(bm, umask));
  ATTN_TRY(check_dm(s, dm));
  if (um && (s->D != 64 || s->dtype == ATTN_F32 || dm)) return ATTN_ERR_UNSUPPORTED;
  ATTN_PTR(q);
  ATTN_PTR(k);
  ATTN_PTR(v);
  ATTN_PTR(out);
  ATTN_PTR(lse);
  ATTN_PTR(dout);
  ATTN_PTR(dq);
  ATTN_PTR(dk);
  ATTN_PTR(dv);
  ATTN_OPT_PTR(key_mask);
  ATTN_TRY(check_ws(ATTN_OP_BWD, s, ws, ws_bytes));
  const void* uk[3] = {nullptr, nullptr, nullptr};
  if (um) ATTN_TRY(user_mod_kernels(um, s->dtype, uk));   // loads the mod's code on this device (first use)
  ATTN_TRY(attn_bwd_preprocess(s, out, lse, dout, key_mask, ws, ws_bytes, stream));
  ATTN_TRY(bwd_dkdv_impl(s, q, k, v, dout, key_mask, dm, bm, mod, scale, dk, dv, ws, ws_bytes, stream, uk[1], umask));
  return bwd_dq_impl(s, q, k, v, dout, key_mask, dm, bm, mod, scale, dq, ws, ws_bytes, stream, uk[2], umask);
}

attn_status attn_bwd_dense(const attn_shape* s, const void* q, const void* k, const void* v, const void* out,
                           const float* lse, const void* dout, const uint8_t* key_mask, const attn_dense_mask* dm,
                           const attn_block_mask* bm, attn_score_mod mod, float scale, void* dq, void* dk, void* dv,
                           void* ws, size_t ws_bytes, attn_stream_t stream) {
  return bwd_all(s, q, k, v, out, lse, dout, key_mask, dm, bm, mod, scale, dq, dk, dv, ws, ws_bytes, stream, nullptr);
}

attn_status attn_bwd_user(const attn_shape* s, const void* q, const void* k, const void* v, const void* out,
                          const float* lse, const void* dout, const uint8_t* key_mask, attn_user_mod um,
                          const attn_block_mask* bm, float scale, void* dq, void* dk, void* dv, void* ws,
                          size_t ws_bytes, attn_stream_t stream) {
  if (!um) return ATTN_ERR_INVALID_ARG;
  return bwd_all(s, q, k, v, out, lse, dout, key_mask, nullptr, bm, ATTN_MOD_NONE, scale, dq, dk, dv, ws, ws_bytes,
                 stream, um);
}

size_t attn_dense_mask_bytes(const attn_shape* s, int bcast_b, int bcast_h) {
  if (!shape_ok(s) || (bcast_b != 0 && bcast_b != 1) || (bcast_h != 0 && bcast_h != 1)) return 0;
  return dense_mask_layout(dense_mask_count(s, bcast_b, bcast_h), s->Sq, s->Skv).total;
}

attn_status attn_pack_dense_mask(const attn_shape* s, const uint8_t* mask, int bcast_b, int bcast_h, void* packed,
                                 size_t packed_bytes, attn_stream_t stream) {
  if (!shape_ok(s) || !mask || !packed || (bcast_b != 0 && bcast_b != 1) || (bcast_h != 0 && bcast_h != 1))
    return ATTN_ERR_INVALID_ARG;
  if (tiles_of(s->Skv) > FWD_MAXKB || tiles_of(s->Sq) > FWD_MAXKB) return ATTN_ERR_SHAPE;
  if (!aligned(packed, 256)) return ATTN_ERR_ALIGN;
  const long long nmask = dense_mask_count(s, bcast_b, bcast_h);
  const DenseMaskLayout l = dense_mask_layout(nmask, s->Sq, s->Skv);
  if (packed_bytes < l.total) return ATTN_ERR_INVALID_ARG;
  uint8_t* base = static_cast<uint8_t*>(packed);
  return cuda_status(launch_dense_mask_pack(mask, nmask, s->Sq, s->Skv, base + l.tiles,
                                            reinterpret_cast<uint32_t*>(base + l.rowbits),
                                            reinterpret_cast<uint32_t*>(base + l.colbits), (cudaStream_t)stream));
}

attn_status attn_decode(const attn_shape* s, const void* q, const void* k, const void* v, const uint8_t* key_mask,
                        attn_score_mod mod, float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                        attn_stream_t stream) {
  if (!shape_ok(s)) return ATTN_ERR_INVALID_ARG;
  if (s->Sq != 1) return ATTN_ERR_SHAPE;
  if (s->D != 64 || s->dtype == ATTN_F32) return ATTN_ERR_UNSUPPORTED;
  ATTN_TRY(check_mod(mod, scale));
  ATTN_PTR(q);
  ATTN_PTR(k);
  ATTN_PTR(v);
  ATTN_PTR(out);
  ATTN_PTR(lse);
  if (key_mask && !aligned(key_mask, 16)) return ATTN_ERR_ALIGN;
  ATTN_TRY(check_ws(ATTN_OP_DECODE, s, ws, ws_bytes));
  const WsLayout w = layout(ATTN_OP_DECODE, s);
  const DecodeSplit d = decode_split(s);
  DecodeParams p;
  std::memset(&p, 0, sizeof(p));
  p.q = q;
  p.k = k;
  p.v = v;
  p.out = out;
  p.lse = lse;
  p.key_mask = key_mask;
  p.partial = at<float>(ws, w.partial);
  p.counter = at<unsigned>(ws, w.counter);
  p.B = s->B;
  p.H = s->H;
  p.Skv = s->Skv;
  p.nsplit = d.nsplit;
  p.keys_per_split = d.kps;
  p.sc = scale * kLog2e;
  p.mod = (int)mod;
  return cuda_status(launch_decode(p, s->dtype == ATTN_BF16, (cudaStream_t)stream));
}

attn_status attn_decode_chunk(const attn_shape* s, const void* q, const void* k, const void* v,
                              const uint8_t* key_mask, attn_score_mod mod, float scale, int q_offset, void* out,
                              float* lse, void* ws, size_t ws_bytes, attn_stream_t stream) {
  if (!shape_ok(s) || q_offset < 0) return ATTN_ERR_INVALID_ARG;
  if (s->D != 64 || s->dtype == ATTN_F32) return ATTN_ERR_UNSUPPORTED;
  if (tiles_of(s->Skv) > FWD_MAXKB || tiles_of(s->Sq) > FWD_MAXKB) return ATTN_ERR_SHAPE;
  ATTN_TRY(check_mod(mod, scale));
  ATTN_PTR(q);
  ATTN_PTR(k);
  ATTN_PTR(v);
  ATTN_PTR(out);
  ATTN_PTR(lse);
  ATTN_OPT_PTR(key_mask);
  ATTN_TRY(check_ws(ATTN_OP_DECODE_CHUNK, s, ws, ws_bytes));
  cudaStream_t st = (cudaStream_t)stream;
  const WsLayout w = layout(ATTN_OP_DECODE_CHUNK, s);
  const ChunkSplit cs = chunk_split(s);
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const long long rq = (long long)s->B * s->H * s->Sq, rk = (long long)s->B * s->H * s->Skv;
  if (!make_tmap(&p.tm_q, q, rq, 64, s->dtype) || !make_tmap(&p.tm_k, k, rk, 64, s->dtype) ||
      !make_tmap(&p.tm_v, v, rk, 64, s->dtype))
    return ATTN_ERR_CUDA;
  p.out = out;
  p.lse = lse;
  p.km = key_mask;   // read as bytes by the kernel's producer: no packing launch
  p.status = at<int>(ws, 0);
  p.B = s->B;
  p.H = s->H;
  p.Sq = s->Sq;
  p.Skv = s->Skv;
  p.nqb = tiles_of(s->Sq);
  p.nkb = tiles_of(s->Skv);
  p.npairs = (p.nqb + 1) / 2;
  p.sc = scale * kLog2e;
  p.timeout_ns = timeout_ns();
  p.q_off = q_offset;
  p.fold = mod_fold_ok(mod, scale, s->H);
  p.inv_scale = scale != 0.f ? 1.f / scale : 0.f;
  p.nsplit = cs.nsplit;
  p.kps = cs.kps;
  p.part = cs.nsplit > 1 ? at<float>(ws, w.partial) : nullptr;
  p.kraw = k;
  p.vraw = v;
  const bool bf16 = s->dtype == ATTN_BF16;
  ATTN_TRY(cuda_status(launch_fwd_d64(p, bf16, (int)mod, st)));
  if (cs.nsplit == 1) return ATTN_OK;   // one kv range: the kernel wrote out and lse itself
  return cuda_status(launch_split_merge(p.part, cs.nsplit, rq, s->Sq, out, lse, bf16, st));
}

attn_status attn_poll_status(void* ws, attn_stream_t stream) {
  if (!ws) return ATTN_ERR_INVALID_ARG;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int word = 0;
  if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return ATTN_ERR_CUDA;
  if (word == 0) return ATTN_OK;
  if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
  return (word & 0xFF) == ATTN_ERR_TIMEOUT ? ATTN_ERR_TIMEOUT : ATTN_ERR_CUDA;
}

}  // extern "C"
