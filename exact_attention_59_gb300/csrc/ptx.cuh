// ptx.cuh - hand-written inline PTX for sm_103a: mbarrier, TMA, tcgen05.
//
// Only the instructions the attention kernels use, each wrapped once.  Every
// wait is bounded by a deadline read from %globaltimer; a wait that runs out
// raises a CTA-wide abort flag in shared memory and writes a status code, so
// all roles of the CTA leave their loops, release tensor memory and return.
#pragma once

#ifdef __CUDACC_RTC__
// Runtime compilation (a user score_mod): no host headers; the fixed-width
// integers and the tensor-map layout that <cstdint> and <cuda.h> give.
typedef unsigned char uint8_t;
typedef unsigned short uint16_t;
typedef unsigned int uint32_t;
typedef unsigned long long uint64_t;
typedef int int32_t;
typedef long long int64_t;
typedef unsigned long long uintptr_t;
typedef struct CUtensorMap_st {
  alignas(64) unsigned long long opaque[16];
} CUtensorMap;
#define INFINITY (__int_as_float(0x7f800000))
#else
#include <cuda.h>
#include <cstdint>
#endif

#define DEVI __device__ __forceinline__

namespace attn {

constexpr int kStatusTimeout = 7;   // ATTN_ERR_TIMEOUT

DEVI uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

DEVI uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

DEVI uint32_t lane_id() { return threadIdx.x & 31u; }

// ---------------------------------------------------------------------------
// Abort / status plumbing
// ---------------------------------------------------------------------------
// A bounded wait's context.  BY_ADDR: the slow paths below take the context's
// address (the context then sits in the thread's stack frame) instead of its
// fields, so a call site passes three words instead of seven.  Which form a
// kernel runs faster with is a matter of measurement: by address helped the
// run-time-compiled score_mod forward and slowed the backward passes.
template <bool BY_ADDR>
struct WaitCtxT {
  volatile int* abort;   // shared memory, CTA-wide
  int* status;           // global status word (workspace offset 0)
  uint64_t timeout_ns;
  int site;              // which wait, recorded in the status word's upper bits
};
using WaitCtx = WaitCtxT<false>;

DEVI void raise_abort(const WaitCtx& c) {
  *c.abort = 1;
  atomicCAS(c.status, 0, kStatusTimeout | (c.site << 8));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
DEVI void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
DEVI void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
DEVI void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

DEVI void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
DEVI void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
DEVI bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// The slow paths of the waits below: a bounded spin that gives up after
// timeout_ns (raising the CTA's abort flag and recording `site` in the status
// word) or as soon as another thread of the CTA has given up.  Kept out of line
// so that the fast path (the phase has already completed) stays small.
static __device__ __noinline__ bool wait_one_slow(uint32_t bar, uint32_t parity, volatile int* abort, int* status,
                                           uint64_t timeout_ns, int site) {
  const uint64_t t0 = global_timer_ns();
  for (;;) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (global_timer_ns() - t0 > timeout_ns) {
      *abort = 1;
      atomicCAS(status, 0, kStatusTimeout | (site << 8));
      return false;
    }
  }
}
static __device__ __noinline__ bool wait_warp_slow(uint32_t bar, uint32_t parity, volatile int* abort, int* status,
                                            uint64_t timeout_ns, int site) {
  uint64_t t0 = 0;
  for (uint32_t it = 0;; ++it) {
    const bool ok = mbar_try_wait(bar, parity);
    if (__all_sync(0xffffffffu, ok)) return true;
    if ((it & 31u) == 31u) {
      int stop = 0;
      if (lane_id() == 0) {
        const uint64_t t = global_timer_ns();
        if (t0 == 0) t0 = t;
        if (*abort) {
          stop = 1;
        } else if (t - t0 > timeout_ns) {
          *abort = 1;
          atomicCAS(status, 0, kStatusTimeout | (site << 8));
          stop = 1;
        }
      }
      if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    }
  }
}

// Waits without honouring the abort flag (bounded by timeout_ns): used on the way
// out, so that copies and MMAs in flight finish before the CTA exits.
DEVI void drain_wait(uint32_t bar, uint32_t parity, uint64_t timeout_ns) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) return;
  }
}

static __device__ __noinline__ bool wait_one_slow_at(uint32_t bar, uint32_t parity, const WaitCtxT<true>* c) {
  return wait_one_slow(bar, parity, c->abort, c->status, c->timeout_ns, c->site);
}
static __device__ __noinline__ bool wait_warp_slow_at(uint32_t bar, uint32_t parity, const WaitCtxT<true>* c) {
  return wait_warp_slow(bar, parity, c->abort, c->status, c->timeout_ns, c->site);
}

// One thread waits for phase `parity` of `bar` to complete.  False = gave up.
template <bool BY_ADDR>
DEVI bool wait_one(uint32_t bar, uint32_t parity, const WaitCtxT<BY_ADDR>& c) {
  if (mbar_try_wait(bar, parity)) return true;
  if constexpr (BY_ADDR) return wait_one_slow_at(bar, parity, &c);
  else return wait_one_slow(bar, parity, c.abort, c.status, c.timeout_ns, c.site);
}

// A whole warp waits; the outcome is warp-uniform (so .sync.aligned tcgen05
// instructions that follow are executed by all 32 lanes together).
template <bool BY_ADDR>
DEVI bool wait_warp(uint32_t bar, uint32_t parity, const WaitCtxT<BY_ADDR>& c) {
  if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;
  if constexpr (BY_ADDR) return wait_warp_slow_at(bar, parity, &c);
  else return wait_warp_slow(bar, parity, c.abort, c.status, c.timeout_ns, c.site);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch and L2 prefetch
// ---------------------------------------------------------------------------
// The grid launched after this one in the stream (with the programmatic
// stream-serialization attribute) may start once every CTA of this grid has
// executed this, or exited.
DEVI void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Blocks until the grids this one depends on have completed and their memory
// operations are visible; returns at once for a grid launched without the attribute.
DEVI void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Asks L2 to fetch [p, p + bytes) from global memory (p 16-byte aligned, bytes a
// multiple of 16); nothing is returned and no completion is tracked.
DEVI void prefetch_l2_bulk(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

// ---------------------------------------------------------------------------
// Thread-block clusters: rank, barrier, distributed shared memory
// ---------------------------------------------------------------------------
DEVI uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Every thread of every CTA of the cluster arrives once per phase, then waits.
DEVI void cluster_arrive_relaxed() { asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory"); }
DEVI void cluster_arrive_release() { asm volatile("barrier.cluster.arrive.release;" ::: "memory"); }
DEVI void cluster_wait_acquire() { asm volatile("barrier.cluster.wait.acquire;" ::: "memory"); }
// Address, in the cluster's shared window, of this CTA's shared-memory address
// `addr` as it lies in the CTA of rank `rank`.
DEVI uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
DEVI void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), 2-D tiles, completion on an mbarrier
// ---------------------------------------------------------------------------
DEVI void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
// c0 = innermost (column, in elements; c0 * elem_size must be a multiple of 16), c1 = row.
DEVI void tma_load_2d(uint32_t dst, const CUtensorMap* m, uint32_t bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::
          "r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar), "r"(c0), "r"(c1)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory, MMA, commit, loads/stores
// ---------------------------------------------------------------------------
DEVI void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
DEVI void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// mbarrier arrives (count 1) once every tcgen05 op issued so far by this thread is done.
DEVI void tc_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (f16 or bf16 inputs, f32 accumulate).
DEVI void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem], kind::f16; A is M x K, 16-bit values packed in pairs per column.
DEVI void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor of kind::f16: f32 accumulator, A/B both f16 (bf16=false) or both bf16.
// a_mn / b_mn: operand stored MN-major (else K-major).
__host__ __device__ constexpr uint32_t idesc_f16(int M, int N, bool bf16, bool a_mn, bool b_mn) {
  return (1u << 4)                                   // D format: f32
         | ((bf16 ? 1u : 0u) << 7)                   // A format
         | ((bf16 ? 1u : 0u) << 10)                  // B format
         | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17)       // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle (tile base 1024-byte aligned).
// K-major: rows of 128 bytes along K, 8-row atoms `sbo` bytes apart (lbo unused).
// MN-major: rows of 128 bytes along MN (64 16-bit values), 8-row K groups `sbo`
// bytes apart, 64-wide MN chunks `lbo` bytes apart.
DEVI uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= 1ull << 46;   // descriptor version for tcgen05
  d |= 2ull << 61;   // SWIZZLE_128B
  return d;
}

// Shared-memory descriptor of a K = 16 operand stored K-major without swizzle:
// 8-row x 16-byte core matrices, the two along K 128 bytes apart (LBO), row
// groups of 8 rows 256 bytes apart (SBO).  Element (row r, k c), c < 16, sits at
// byte (r / 8) * 256 + (c / 8) * 128 + (r % 8) * 16 + (c % 8) * 2: 4 KB for 128 rows.
DEVI uint32_t k16_offset(int r, int c) {
  return (uint32_t)(r >> 3) * 256u + (uint32_t)(c >> 3) * 128u + (uint32_t)(r & 7) * 16u + (uint32_t)(c & 7) * 2u;
}
// The same layout with a stride of 0 between 8-row groups: every group of 8
// rows of the operand reads the one group at saddr (256 bytes), an operand
// whose rows repeat with period 8.
DEVI uint64_t sdesc_k16_rows8(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(128u >> 4) << 16;
  d |= 1ull << 46;
  return d;
}
DEVI uint64_t sdesc_k16(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>(128u >> 4) << 16;
  d |= static_cast<uint64_t>(256u >> 4) << 32;
  d |= 1ull << 46;   // descriptor version for tcgen05; layout type 0 = no swizzle
  return d;
}

// tcgen05.ld 32x32b: each lane of the warp reads its own TMEM lane, 32 consecutive
// 32-bit columns.  The wait is in the same statement, so the values are ready on return.
DEVI void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
}

DEVI void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

// Wider forms of the same 32x32b loads and stores (one instruction, one wait).
DEVI void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr)
      : "memory");
}
DEVI void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x128.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]), "=r"(r[64]), "=r"(r[65]), "=r"(r[66]), "=r"(r[67]), "=r"(r[68]), "=r"(r[69]), "=r"(r[70]), "=r"(r[71]), "=r"(r[72]), "=r"(r[73]), "=r"(r[74]), "=r"(r[75]), "=r"(r[76]), "=r"(r[77]), "=r"(r[78]), "=r"(r[79]), "=r"(r[80]), "=r"(r[81]), "=r"(r[82]), "=r"(r[83]), "=r"(r[84]), "=r"(r[85]), "=r"(r[86]), "=r"(r[87]), "=r"(r[88]), "=r"(r[89]), "=r"(r[90]), "=r"(r[91]), "=r"(r[92]), "=r"(r[93]), "=r"(r[94]), "=r"(r[95]), "=r"(r[96]), "=r"(r[97]), "=r"(r[98]), "=r"(r[99]), "=r"(r[100]), "=r"(r[101]), "=r"(r[102]), "=r"(r[103]), "=r"(r[104]), "=r"(r[105]), "=r"(r[106]), "=r"(r[107]), "=r"(r[108]), "=r"(r[109]), "=r"(r[110]), "=r"(r[111]), "=r"(r[112]), "=r"(r[113]), "=r"(r[114]), "=r"(r[115]), "=r"(r[116]), "=r"(r[117]), "=r"(r[118]), "=r"(r[119]), "=r"(r[120]), "=r"(r[121]), "=r"(r[122]), "=r"(r[123]), "=r"(r[124]), "=r"(r[125]), "=r"(r[126]), "=r"(r[127])
      : "r"(taddr)
      : "memory");
}
DEVI void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]), "r"(r[32]), "r"(r[33]), "r"(r[34]), "r"(r[35]), "r"(r[36]), "r"(r[37]), "r"(r[38]), "r"(r[39]), "r"(r[40]), "r"(r[41]), "r"(r[42]), "r"(r[43]), "r"(r[44]), "r"(r[45]), "r"(r[46]), "r"(r[47]), "r"(r[48]), "r"(r[49]), "r"(r[50]), "r"(r[51]), "r"(r[52]), "r"(r[53]), "r"(r[54]), "r"(r[55]), "r"(r[56]), "r"(r[57]), "r"(r[58]), "r"(r[59]), "r"(r[60]), "r"(r[61]), "r"(r[62]), "r"(r[63]) : "memory");
}

DEVI void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------------------
// Packed two-float arithmetic (sm_100+): one instruction for two lanes of data
// ---------------------------------------------------------------------------
DEVI uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
DEVI void unf2(uint64_t v, float& lo, float& hi) { asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v)); }
DEVI uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
  return r;
}
DEVI uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
DEVI uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t r;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
  return r;
}
DEVI float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// ---------------------------------------------------------------------------
// Arithmetic helpers
// ---------------------------------------------------------------------------
DEVI float ex2(float x) {   // MUFU 2^x; 2^-inf = 0
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
DEVI float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Packs (lo, hi) into one 32-bit word of two 16-bit floats, round to nearest even.
template <bool BF16>
DEVI uint32_t pack2(float lo, float hi) {
  uint32_t r;
  if constexpr (BF16)
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
template <bool BF16>
DEVI float2 unpack2(uint32_t w) {
  float2 f;
  if constexpr (BF16) {
    f.x = __uint_as_float(w << 16);
    f.y = __uint_as_float(w & 0xFFFF0000u);
  } else {
    unsigned short lo = static_cast<unsigned short>(w & 0xFFFFu), hi = static_cast<unsigned short>(w >> 16);
    asm("cvt.f32.f16 %0, %1;" : "=f"(f.x) : "h"(lo));
    asm("cvt.f32.f16 %0, %1;" : "=f"(f.y) : "h"(hi));
  }
  return f;
}

// One value rounded to the 16-bit type (round to nearest even), and back.
template <bool BF16>
DEVI uint16_t to16(float x) { return static_cast<uint16_t>(pack2<BF16>(x, 0.f) & 0xFFFFu); }
template <bool BF16>
DEVI float from16(uint16_t v) { return unpack2<BF16>(static_cast<uint32_t>(v)).x; }

// Word of the packed key mask (bit j = key 32 w + j kept) holding key `key` of
// batch b; words past the end of the row (a partial last kv block) read as 0.
DEVI uint32_t km_word(const uint32_t* bits, int b, int Skv, int key) {
  const int nw = (Skv + 31) >> 5, wi = key >> 5;
  return wi < nw ? __ldg(bits + (size_t)b * nw + wi) : 0u;
}

// One f32 value x as three 16-bit terms, x = t0 + t1 + 2048 t2, written to columns
// 0..2 of row r of a K = 16 operand (no swizzle).  The 2048 t2 term keeps f16 in
// range; t0 + t1 carry the rest to about 2^-22 relative.  An infinity goes to t2
// alone (-inf for a row with no kept key; +inf when a negative scale divided it).
template <bool BF16>
DEVI void split3(float x, uint8_t* op, int r) {
  float a2, a0, a1;
  if (fabsf(x) == INFINITY) {
    a2 = x;
    a0 = a1 = 0.f;
  } else {
    a2 = from16<BF16>(to16<BF16>(x * (1.f / 2048.f)));
    const float r1 = x - 2048.f * a2;
    a0 = from16<BF16>(to16<BF16>(r1));
    a1 = r1 - a0;
  }
  *reinterpret_cast<uint16_t*>(op + k16_offset(r, 0)) = to16<BF16>(a0);
  *reinterpret_cast<uint16_t*>(op + k16_offset(r, 1)) = to16<BF16>(a1);
  *reinterpret_cast<uint16_t*>(op + k16_offset(r, 2)) = to16<BF16>(a2);
}

// x as three 16-bit terms t0 + t1 + t2 (each the rounded remainder of the
// previous ones): about 3 x 8 significant bits in bf16, 3 x 11 in f16.  For
// finite values of moderate size (|x| well inside the 16-bit range).
template <bool BF16>
DEVI void split3_plain(float x, uint16_t (&t)[3]) {
  t[0] = to16<BF16>(x);
  const float r1 = x - from16<BF16>(t[0]);
  t[1] = to16<BF16>(r1);
  t[2] = to16<BF16>(r1 - from16<BF16>(t[1]));
}

}  // namespace attn
