/*
 * attn.h - C ABI of a GB300 (sm_103a) exact softmax attention library.
 *
 * The operation is the tiled, IO-aware exact attention of FlashAttention
 * (Dao et al. 2022, cited by the attnax Pallas kernel page, "FlashAttention
 * forward pass compiled with Pallas"): per query row,
 *     S = scale * q K^T + score_mod bias,  masked entries = -inf,
 *     P = softmax(S),  O = P V,  lse = log sum_j exp(S_j),
 * computed with the online-softmax recurrence of the attnax Pallas kernel body
 * (running max m, running sum l, accumulator rescaled by exp(m_old - m_new)),
 * plus the FlexAttention-style hooks of the flaxattention README ("Example
 * usage": score_mod, create_block_mask(causal_mask, ...)) and the key-padding
 * mask of shape (batch, seq) of the flash-attention-jax docs ("3. Use
 * flash_attention").
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Tensors are caller-owned DEVICE memory, BHSD contiguous:
 *      q (B, H, Sq, D), k and v (B, H, Skv, D), out/dout/dq (B, H, Sq, D),
 *      dk/dv (B, H, Skv, D), all in the dtype of attn_shape.dtype;
 *      lse (B, H, Sq) float32, natural log (the second return value of
 *      flash_attention, read as the row log-sum-exp).
 *    This is the (batch, heads, seq, dim) layout of the attnax Pallas
 *    forward's arguments.
 *  - key_mask is uint8 (B, Skv), nonzero = attend; NULL = no key mask.
 *  - Every pointer must be 16-byte aligned (the TMA engine needs it), else
 *    ATTN_ERR_ALIGN.
 *  - Prefill (attn_fwd / attn_bwd) with D = 64 (f16, bf16 and f32) takes any
 *    Sq, Skv >= 1 (up to 2048 tiles of 128): the last q and kv tiles may be
 *    partial; keys past Skv get no weight and rows past Sq are not written.
 *    D = 512 needs Sq and Skv to be multiples of 128, as the attnax Pallas
 *    forward requires seq_q % block_q == 0 and seq_kv % block_kv == 0 with
 *    block_q = block_kv = 128; else ATTN_ERR_SHAPE.  D must be 64 (all
 *    dtypes) or 512 (bf16/f16, forward and backward).
 *  - float32 runs on the tensor cores too: each contraction as three TF32
 *    products (hi x hi + hi x lo + lo x hi of the TF32 parts), f32 accumulate.
 *  - The library allocates no memory and keeps no state.  Scratch space
 *    ("workspace") is caller-owned device memory of attn_workspace_size()
 *    bytes, 256-byte aligned, and must be zero-filled before its first use
 *    (its first word is the status word, below; the item counters of the
 *    forward and of the two backward passes, which every call leaves at
 *    zero, lie in its first 256 bytes too); any call and shape may use it
 *    after that (completion tickets are zeroed by the call that uses them,
 *    with an asynchronous memset on `stream`).  Calls on one workspace must
 *    not overlap in time (use one workspace per stream).
 *  - Calls are asynchronous on `stream` and never synchronise, except
 *    attn_poll_status().  Arguments are validated before anything is
 *    launched: a call that returns an error has launched nothing.
 *  - Device-side waits are bounded (ATTN_TIMEOUT_NS environment variable,
 *    default 2 s).  A kernel whose wait runs out stops, writes
 *    ATTN_ERR_TIMEOUT into the workspace status word and returns; read it
 *    with attn_poll_status().
 *  - Masked scores are -inf: a row with no kept key gets O = 0, lse = -inf
 *    and zero gradients.
 *  - `scale` multiplies q k^T; it must be finite and nonzero (negative is
 *    allowed), else ATTN_ERR_INVALID_ARG.  The pages use 1/sqrt(D).
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream; the same handle as cudaStream_t / CUstream.  NULL = legacy default stream. */
typedef struct CUstream_st* attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* NULL pointer, negative size, bad enum, bad scale */
  ATTN_ERR_SHAPE = 2,       /* Sq/Skv not a multiple of 128 (f32 or D=512 prefill), more than 2048 tiles,
                               Sq != 1 (decode), size overflow */
  ATTN_ERR_ALIGN = 3,       /* a pointer is not 16-byte aligned (workspace: 256-byte) */
  ATTN_ERR_UNSUPPORTED = 4, /* dtype / D / mod / block-size combination not built */
  ATTN_ERR_WORKSPACE = 5,   /* workspace NULL or smaller than attn_workspace_size() */
  ATTN_ERR_CUDA = 6,        /* a CUDA runtime call or kernel launch failed */
  ATTN_ERR_TIMEOUT = 7      /* a device-side wait ran out (reported by attn_poll_status) */
} attn_status;

typedef enum { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 } attn_dtype;

/* score_mod hooks (flaxattention README "Example usage"; attnax Pallas kernel
 * body applies score_mod(scores, b, h, q_idx, kv_idx) with global indices after
 * the scale and before the mask).  h is 0-based.
 *   NONE          no change
 *   ALIBI         + slope_h * (kv_idx - q_idx),  slope_h = 2^(-8 (h+1) / H)
 *   CHECKERBOARD  + 0.5 if (q_idx + kv_idx) is even, else - 0.5
 *   CAUSAL        -inf where kv_idx > q_idx (no tile skipping by itself)   */
typedef enum {
  ATTN_MOD_NONE = 0,
  ATTN_MOD_ALIBI = 1,
  ATTN_MOD_CHECKERBOARD = 2,
  ATTN_MOD_CAUSAL = 3
} attn_score_mod;

/* mask_mod of a block mask (flaxattention README: create_block_mask(causal_mask, ...)).
 * ATTN_MASKMOD_USER: the mask expression of the run-time-compiled user mod
 * given with the call (attn_fwd_user / attn_bwd_user only; see
 * attn_user_mod_create_masked), which built the tile states. */
typedef enum { ATTN_MASKMOD_NONE = 0, ATTN_MASKMOD_CAUSAL = 1, ATTN_MASKMOD_USER = 2 } attn_mask_mod;

/* Block-mask tile states. */
enum { ATTN_TILE_EMPTY = 0, ATTN_TILE_PARTIAL = 1, ATTN_TILE_FULL = 2 };

typedef enum { ATTN_OP_FWD = 0, ATTN_OP_BWD = 1, ATTN_OP_DECODE = 2, ATTN_OP_DECODE_CHUNK = 3 } attn_op;

typedef struct {
  int B, H, Sq, Skv, D;
  attn_dtype dtype;
} attn_shape;

/* Block mask: one uint8 state per (q-block, kv-block) tile, laid out
 * (bcast_b ? 1 : B, bcast_h ? 1 : H, ceil(Sq/block_q), ceil(Skv/block_kv)),
 * row-major, device memory.  EMPTY tiles are skipped (all entries masked),
 * PARTIAL tiles apply mask_mod elementwise, FULL tiles are kept whole.
 * block_q = block_kv = 128 is the only size built. */
typedef struct {
  const uint8_t* tiles;
  int bcast_b, bcast_h;
  int block_q, block_kv;
  attn_mask_mod mask_mod;
} attn_block_mask;

/* Dense (query, key) mask, as the attnax pallas_flash_attention arguments
 * take it: a boolean mask broadcastable to (batch, heads, seq_q, seq_kv).
 * Here: uint8 (bcast_b ? 1 : B, bcast_h ? 1 : H, Sq, Skv), row-major device
 * memory, nonzero = attend; it is combined (AND) with the key mask, the
 * score_mod and the block mask.  attn_pack_dense_mask turns it once into
 * the packed form the kernels read (row bits, column bits and one state
 * per 128 x 128 tile; tiles with no kept pair are skipped, tiles with every
 * pair kept are not tested per entry); the packed form can be reused by any
 * number of forward and backward calls of the same shape.  Taken on the
 * D = 64 path, every dtype (ATTN_ERR_UNSUPPORTED at D = 512). */
typedef struct {
  const void* packed;    /* device, 256-byte aligned, written by attn_pack_dense_mask */
  size_t packed_bytes;   /* its size: at least attn_dense_mask_bytes() */
  int bcast_b, bcast_h;  /* 0 or 1, as given to attn_pack_dense_mask */
} attn_dense_mask;

/* Bytes of workspace that `op` needs for `shape` (0 if the shape is invalid).
 * Monotonic non-decreasing in every dimension of the shape. */
size_t attn_workspace_size(attn_op op, const attn_shape* shape);

/* Builds block-mask tile states on the device: the analogue of
 * create_block_mask(mask_mod, B, H, Sq, Skv) in the flaxattention README.
 * tiles: device uint8 (B, H, ceil(Sq/bq), ceil(Skv/bkv)).  A tile is FULL
 * when mask_mod keeps all its entries, EMPTY when it keeps none, else PARTIAL. */
attn_status attn_build_block_mask(attn_mask_mod mask_mod, int B, int H, int Sq, int Skv, int bq,
                                  int bkv, uint8_t* tiles, attn_stream_t stream);

/* Bytes of the packed form of a dense mask for `shape` (B, H, Sq, Skv are
 * used) with the given broadcast flags; 0 if an argument is invalid. */
size_t attn_dense_mask_bytes(const attn_shape* shape, int bcast_b, int bcast_h);

/* Packs a dense uint8 mask (layout in attn_dense_mask) into `packed`
 * (caller-owned device memory, 256-byte aligned, at least
 * attn_dense_mask_bytes() bytes), asynchronously on `stream`.  The mask
 * itself needs no alignment (16-byte aligned rows with Skv % 16 == 0 are
 * read 16 bytes at a time).  Errors: ATTN_ERR_INVALID_ARG (NULL pointer,
 * flag not 0/1, packed too small), ATTN_ERR_SHAPE (more than 2048 tiles of
 * 128 along Sq or Skv), ATTN_ERR_ALIGN (packed). */
attn_status attn_pack_dense_mask(const attn_shape* shape, const uint8_t* mask, int bcast_b, int bcast_h,
                                 void* packed, size_t packed_bytes, attn_stream_t stream);

/* Forward: out = softmax(mask(scale q k^T + mod)) v and lse (attnax Pallas
 * kernel body, online softmax with exp2/log2 arithmetic as in the
 * flaxattention README's "log2 trick").
 *   key_mask: nullable; bm: nullable (NULL = no block mask);
 *   debug_visited: nullable uint8 (B, H, Sq/128, Skv/128); when given, each
 *   entry is set to 1 if the kernel computed that tile and 0 if it skipped it.
 *   D = 512 is built for f16/bf16 (key mask, block mask and the built-in
 *   mods; Sq, Skv multiples of 128). */
attn_status attn_fwd(const attn_shape* shape, const void* q, const void* k, const void* v,
                     const uint8_t* key_mask, const attn_block_mask* bm, attn_score_mod mod,
                     float scale, void* out, float* lse, void* ws, size_t ws_bytes,
                     attn_stream_t stream, uint8_t* debug_visited);

/* attn_fwd with a dense (query, key) mask `dm` (nullable; NULL = attn_fwd).
 * The visited map also leaves out tiles with no pair kept by dm.  Errors as
 * attn_fwd, plus ATTN_ERR_INVALID_ARG (dm->packed NULL, flag not 0/1,
 * packed_bytes too small), ATTN_ERR_ALIGN (dm->packed) and
 * ATTN_ERR_UNSUPPORTED (D = 512). */
attn_status attn_fwd_dense(const attn_shape* shape, const void* q, const void* k, const void* v,
                           const uint8_t* key_mask, const attn_dense_mask* dm, const attn_block_mask* bm,
                           attn_score_mod mod, float scale, void* out, float* lse, void* ws,
                           size_t ws_bytes, attn_stream_t stream, uint8_t* debug_visited);

/* Backward of sum(dout * out): dq, dk, dv (same shapes and dtype as q, k, v).
 * Takes the forward's out and lse and the same key_mask, bm, mod and scale.
 * Runs three kernels: a preprocess (D_i = rowsum(dout * out)), a dK/dV pass
 * over kv blocks and a dQ pass over q blocks; no atomics, so results are
 * bitwise reproducible.  D = 64 (all dtypes) and 512 (f16/bf16). */
attn_status attn_bwd(const attn_shape* shape, const void* q, const void* k, const void* v,
                     const void* out, const float* lse, const void* dout,
                     const uint8_t* key_mask, const attn_block_mask* bm, attn_score_mod mod,
                     float scale, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                     attn_stream_t stream);

/* attn_bwd with the forward's dense mask `dm` (nullable; NULL = attn_bwd);
 * errors as attn_fwd_dense. */
attn_status attn_bwd_dense(const attn_shape* shape, const void* q, const void* k, const void* v,
                           const void* out, const float* lse, const void* dout, const uint8_t* key_mask,
                           const attn_dense_mask* dm, const attn_block_mask* bm, attn_score_mod mod,
                           float scale, void* dq, void* dk, void* dv, void* ws, size_t ws_bytes,
                           attn_stream_t stream);

/* The three phases of attn_bwd as separate calls, in this order, on one
 * workspace (for timing a phase alone).  Same arguments as attn_bwd. */
attn_status attn_bwd_preprocess(const attn_shape* shape, const void* out, const float* lse,
                                const void* dout, const uint8_t* key_mask, void* ws,
                                size_t ws_bytes, attn_stream_t stream);
attn_status attn_bwd_dkdv(const attn_shape* shape, const void* q, const void* k, const void* v,
                          const void* dout, const uint8_t* key_mask, const attn_block_mask* bm,
                          attn_score_mod mod, float scale, void* dk, void* dv, void* ws,
                          size_t ws_bytes, attn_stream_t stream);
attn_status attn_bwd_dq(const attn_shape* shape, const void* q, const void* k, const void* v,
                        const void* dout, const uint8_t* key_mask, const attn_block_mask* bm,
                        attn_score_mod mod, float scale, void* dq, void* ws, size_t ws_bytes,
                        attn_stream_t stream);

/* Single-query decode (shape->Sq must be 1; q_idx = 0): split-KV partial
 * softmax per (b, h, split), K and V streamed straight into registers with
 * 16-byte loads in rounds of 128 keys per split, the splits of a (b, h)
 * merged in the same launch: within a thread-block cluster of up to 8 splits
 * through distributed shared memory, across the clusters of a long (b, h)
 * through the workspace by the last cluster to finish (flaxattention README
 * "Decoding").  f16/bf16, D = 64.  The kernel is launched with programmatic
 * dependent launch: it may start while the previous kernel in `stream`
 * drains, but reads q, k, v, the key mask and writes anything only after that
 * kernel has completed, so stream order holds as for any launch.  Its only
 * waits are cluster barriers among CTAs that run together and always reach
 * them (no spin on memory), so it has no timeout to report. */
attn_status attn_decode(const attn_shape* shape, const void* q, const void* k, const void* v,
                        const uint8_t* key_mask, attn_score_mod mod, float scale, void* out,
                        float* lse, void* ws, size_t ws_bytes, attn_stream_t stream);

/* attn_decode without a caller workspace, for callers that cannot allocate
 * device memory: for example an operator running inside a host framework
 * that owns all device memory and offers no allocation hook, or a serving
 * loop whose memory plan is fixed at start-up and must not call cudaMalloc
 * (directly or through a caching allocator) while it serves.  The pages have
 * no counterpart of this entry point; it exists for those callers only.
 *   - Same arguments, layout and result as attn_decode (f16/bf16, D = 64,
 *     Sq = 1), minus ws and ws_bytes.  It allocates nothing: its scratch is a
 *     4 MiB array built into the library, which every GPU that loads the
 *     library holds until the process exits.
 *   - Shapes whose scratch (B*H*nsplit*(D+2)*4 bytes of partials plus B*H*4
 *     bytes of tickets) exceeds 4 MiB are rejected with ATTN_ERR_WORKSPACE.
 *   - It runs on the CURRENT device; `stream` must belong to it.  Every call
 *     looks up the array's device address there (cudaGetSymbolAddress); the
 *     first call on a device also loads the library's device code on it, so
 *     make that first call before any stream capture.
 *   - Like attn_decode, its kernel spins on no memory word (its only waits
 *     are cluster barriers), so there is no timeout to report and no status
 *     word.
 *   - Every call on a device shares the one array.  A call whose (b, h)
 *     rows need more than one cluster of splits (more than 4096 keys) zeroes
 *     the tickets it uses with an asynchronous memset on `stream` first.
 *     Calls that overlap in time on the GPU (other streams, other threads)
 *     race on the array and give wrong results: serialise them. */
attn_status attn_decode_noalloc(const attn_shape* shape, const void* q, const void* k, const void* v,
                                const uint8_t* key_mask, attn_score_mod mod, float scale, void* out,
                                float* lse, attn_stream_t stream);

/* Decode of a chunk of shape->Sq >= 1 queries against a KV cache of Skv keys
 * that already holds earlier tokens: query row i sits at position
 * q_offset + i, the position every score_mod uses (the causal rule keeps
 * keys kv <= q_offset + i; ALiBi and checkerboard see the position).  The
 * flaxattention README's "Decoding" benchmark and its "faster decoding"
 * item cover q_len = 1; this is the same computation for a few queries
 * (speculative or chunked decoding), run on the tensor cores: the kv blocks
 * are split over about one CTA per SM and a second launch merges the
 * per-split rows.  f16/bf16, D = 64, any Sq and Skv (ATTN_ERR_SHAPE past
 * 2048 tiles of 128), optional key_mask; no block or dense mask.
 * Workspace: attn_workspace_size(ATTN_OP_DECODE_CHUNK, shape).
 * Errors: ATTN_ERR_INVALID_ARG (q_offset < 0, NULL pointer, bad mod or
 * scale), ATTN_ERR_UNSUPPORTED (f32 or D != 64), ATTN_ERR_ALIGN,
 * ATTN_ERR_WORKSPACE. */
attn_status attn_decode_chunk(const attn_shape* shape, const void* q, const void* k, const void* v,
                              const uint8_t* key_mask, attn_score_mod mod, float scale, int q_offset, void* out,
                              float* lse, void* ws, size_t ws_bytes, attn_stream_t stream);

/* A score_mod compiled at run time (NVRTC): the flaxattention README's hooks
 * take arbitrary callables, the enum above covers the ones it names.  Here a
 * user score_mod is a C expression for an additive bias in the int
 * variables b, h, q, kv (q and kv are positions; -INFINITY masks the pair):
 * score' = score + bias, the form of every mod the pages name, so the
 * backward needs no derivative of it.  It is compiled into the D = 64
 * forward, dK/dV and dQ kernels for one 16-bit dtype (about 2 s, no GPU
 * needed); the result is loaded on a device when a call first uses it there.
 * The expression runs as device code in the caller's process.
 *   log: nullable buffer for the compiler's messages (also on success).
 * Errors: ATTN_ERR_INVALID_ARG (NULL, empty or over 4096 characters, or the
 * expression does not compile: see log), ATTN_ERR_UNSUPPORTED (f32, or the
 * kernel sources are not beside the library). */
typedef struct attn_user_mod_st* attn_user_mod;
attn_status attn_user_mod_create(const char* bias_expr, attn_dtype dtype, attn_user_mod* mod, char* log,
                                 size_t log_bytes);
/* A user score_mod with a user mask_mod (flaxattention README "Example usage":
 * create_block_mask(mask_mod, B, H, Sq, Skv) takes any mask function and
 * FlexAttention skips the tiles it empties).  mask_expr is a C expression in
 * the int variables b, h, q, kv (positions), nonzero = the query attends to
 * the key; bias_expr (nullable or empty: no bias) is as in
 * attn_user_mod_create.  Besides the forward, dK/dV and dQ kernels the mod
 * then holds a block-mask builder (attn_build_block_mask_user).  A block mask
 * with mask_mod = ATTN_MASKMOD_USER, passed with this mod to attn_fwd_user /
 * attn_bwd_user, skips EMPTY tiles, takes FULL tiles whole and evaluates
 * mask_expr on every entry of a PARTIAL tile: the tiles must come from the
 * same mod.  Errors as attn_user_mod_create (ATTN_ERR_INVALID_ARG also when
 * both expressions are NULL or empty). */
attn_status attn_user_mod_create_masked(const char* bias_expr, const char* mask_expr, attn_dtype dtype,
                                        attn_user_mod* mod, char* log, size_t log_bytes);

/* Tile states of `mod`'s mask expression (the analogue of create_block_mask
 * with a user mask function): tiles is device uint8 (B, H, ceil(Sq/bq),
 * ceil(Skv/bkv)); a tile is FULL when the expression keeps every in-range
 * (q, kv) of it, EMPTY when it keeps none, else PARTIAL.  Asynchronous on
 * `stream` (the current device).  bq = bkv = 128 only (ATTN_ERR_UNSUPPORTED
 * otherwise); ATTN_ERR_INVALID_ARG for a NULL pointer, a non-positive size or
 * a mod without a mask expression. */
attn_status attn_build_block_mask_user(attn_user_mod mod, int B, int H, int Sq, int Skv, int bq, int bkv,
                                       uint8_t* tiles, attn_stream_t stream);

/* Frees a user score_mod (NULL is ignored).  Waits for all work on each
 * device the mod was loaded on before unloading its code, so a call still
 * queued on a stream finishes first; it must not race with a new call. */
void attn_user_mod_destroy(attn_user_mod mod);

/* attn_fwd / attn_bwd with a user score_mod in place of the enum (f16/bf16,
 * D = 64, the dtype the mod was built for, else ATTN_ERR_UNSUPPORTED); the
 * key mask, block mask and debug_visited work as in attn_fwd.  Errors as
 * attn_fwd. */
attn_status attn_fwd_user(const attn_shape* shape, const void* q, const void* k, const void* v,
                          const uint8_t* key_mask, attn_user_mod mod, const attn_block_mask* bm, float scale,
                          void* out, float* lse, void* ws, size_t ws_bytes, attn_stream_t stream,
                          uint8_t* debug_visited);
attn_status attn_bwd_user(const attn_shape* shape, const void* q, const void* k, const void* v, const void* out,
                          const float* lse, const void* dout, const uint8_t* key_mask, attn_user_mod mod,
                          const attn_block_mask* bm, float scale, void* dq, void* dk, void* dv, void* ws,
                          size_t ws_bytes, attn_stream_t stream);

/* Synchronises `stream`, then reads and clears the workspace status word.
 * Returns ATTN_OK, ATTN_ERR_TIMEOUT (a device wait ran out), or
 * ATTN_ERR_CUDA (the stream reported an error). */
attn_status attn_poll_status(void* ws, attn_stream_t stream);

/* Static text for a status code. */
const char* attn_status_string(attn_status s);

#ifdef __cplusplus
}
#endif
#endif /* ATTN_GB300_H */
