// tc.cuh -- thin inline-PTX wrappers for sm_100-family features used by the
// tensor-core kernels: mbarriers with bounded waits, TMA tile loads, tcgen05
// (TMEM allocation, MMA, commit, TMEM loads) and 128-byte-swizzled shared
// memory operand tiles.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {
namespace tc {

__device__ __forceinline__ uint32_t pack_bf16(float lo_elem, float hi_elem);
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t &hi, uint32_t &lo);

// Time limit of every mbarrier wait (ns of %globaltimer); on expiry the kernel
// records where it gave up in the device error record and unwinds instead of
// spinning forever.
constexpr uint64_t WAIT_NS = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
// The 1024-byte-aligned start of the dynamic shared memory, formed by pointer arithmetic on the shared
// array itself so that the compiler keeps its address space: plain C++ loads and stores through it stay
// shared-memory instructions (an integer round trip would make them generic ones).
__device__ __forceinline__ unsigned char *smem_align1024(unsigned char *raw) {
    return raw + ((1024u - (smem_u32(raw) & 1023u)) & 1023u);
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(bar) : "memory");
}
// One arrival for the whole warp: every lane's prior memory operations (and fences) are ordered before
// lane 0's arrival by the __syncwarp.  Barriers fed this way count warps, not threads.
__device__ __forceinline__ void mbar_arrive_warp(uint32_t bar) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}
// Non-blocking probe: true once the phase with the given parity has completed.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Potentially blocking probe: the hardware may park the warp until the phase
// completes or a short system-defined interval elapses.
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait.  Returns false if the barrier did not complete within limit_ns
// or another thread already raised *abort; on its own expiry it raises *abort.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          uint64_t limit_ns = WAIT_NS) {
    if (mbar_test(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        if (mbar_try(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > limit_ns) {
            *abort = 1;
            return false;
        }
    }
}
// Warp-uniform result of a bounded wait (tcgen05.ld and other .sync.aligned
// instructions after it need every lane of the warp).
__device__ __forceinline__ bool mbar_wait_warp(uint32_t bar, uint32_t parity, volatile int *abort,
                                               uint64_t limit_ns = WAIT_NS) {
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort, limit_ns));
}
// Bounded wait without an abort flag (used for draining at exit).
__device__ __forceinline__ bool mbar_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns = WAIT_NS) {
    const uint64_t t0 = global_ns();
    while (!mbar_test(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// ------------------------------------------------------------------ fences
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
// Named barrier that also ANDs a predicate over the participating threads, so a
// group leaves a loop together (nobody is left waiting at the next bar.sync).
__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
        "[%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}
// Plain (untiled) bulk copy global -> shared; both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar)
                 : "memory");
}
// Plain bulk copy shared -> global (same alignment rules), tracked by the issuing thread's bulk groups.
__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(reinterpret_cast<uint64_t>(dst)),
                 "r"(src), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// The issuing thread's committed bulk stores have read their shared-memory sources (free for reuse).
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// The issuing thread's committed bulk stores have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (bf16 in, fp32 accumulate), one CTA.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05 operations of this thread complete.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}

// Instruction descriptor, kind::f16: fp32 D, bf16 A and B; a_mn / b_mn select
// MN-major (transposed) operands.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t addr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// TMEM loads and stores.  tcgen05.ld fills its destination registers asynchronously and tcgen05.st
// may read its source registers after it issues; both are complete only at the matching tcgen05.wait.
// Each wrapper below issues its loads (or stores) AND the wait in ONE asm statement: the compiler sees
// the destination registers defined (and the source registers used) only once the wait has completed,
// so it can neither read, spill nor reuse them early.  (With the wait in a separate statement the
// compiler may legally spill a destination register in between, which stores an unfinished value.)
#define GDN_R8(o) "=r"(r[o]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]), "=r"(r[o + 5]), \
    "=r"(r[o + 6]), "=r"(r[o + 7])
#define GDN_S8(o) "=r"(s[o]), "=r"(s[o + 1]), "=r"(s[o + 2]), "=r"(s[o + 3]), "=r"(s[o + 4]), "=r"(s[o + 5]), \
    "=r"(s[o + 6]), "=r"(s[o + 7])
#define GDN_I8(a, o) "r"(a[o]), "r"(a[o + 1]), "r"(a[o + 2]), "r"(a[o + 3]), "r"(a[o + 4]), "r"(a[o + 5]), \
    "r"(a[o + 6]), "r"(a[o + 7])

// 32 lanes x 32 consecutive columns of 32-bit TMEM cells -> 32 registers per thread (waited).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GDN_R8(0), GDN_R8(8), GDN_R8(16), GDN_R8(24)
        : "r"(taddr)
        : "memory");
}
// 32 lanes x 16 consecutive columns -> 16 registers per thread (waited).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GDN_R8(0), GDN_R8(8)
        : "r"(taddr)
        : "memory");
}
// Two 16-column loads in flight together (waited).
__device__ __forceinline__ void tmem_ld16x2(uint32_t ta, uint32_t (&r)[16], uint32_t tb, uint32_t (&s)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%32];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, "
        "%29, %30, %31}, [%33];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GDN_R8(0), GDN_R8(8), GDN_S8(0), GDN_S8(8)
        : "r"(ta), "r"(tb)
        : "memory");
}
// Two 8-column loads, waited.
__device__ __forceinline__ void tmem_ld8x2(uint32_t ta, uint32_t (&r)[8], uint32_t tb, uint32_t (&s)[8]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%16];\n\t"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8, %9, %10, %11, %12, %13, %14, %15}, [%17];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GDN_R8(0), GDN_S8(0)
        : "r"(ta), "r"(tb)
        : "memory");
}
// Two 16-column stores (e.g. a hi / lo pair), waited.
__device__ __forceinline__ void tmem_st16x2(uint32_t ta, const uint32_t (&a)[16], uint32_t tb,
                                            const uint32_t (&b)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%1], {%18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
        "%30, %31, %32, %33};\n\t"
        "tcgen05.wait::st.sync.aligned;"
        :
        : "r"(ta), "r"(tb), GDN_I8(a, 0), GDN_I8(a, 8), GDN_I8(b, 0), GDN_I8(b, 8)
        : "memory");
}
// Two 8-column stores, waited.
__device__ __forceinline__ void tmem_st8x2(uint32_t ta, const uint32_t (&a)[8], uint32_t tb, const uint32_t (&b)[8]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%2, %3, %4, %5, %6, %7, %8, %9};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x8.b32 [%1], {%10, %11, %12, %13, %14, %15, %16, %17};\n\t"
        "tcgen05.wait::st.sync.aligned;"
        :
        : "r"(ta), "r"(tb), GDN_I8(a, 0), GDN_I8(b, 0)
        : "memory");
}
#undef GDN_R8
#undef GDN_S8
#undef GDN_I8
// D[tmem] (+)= A[tmem] * B[smem]^T; A: 128 lanes, 16 bf16 per k-step packed in 8 columns.
__device__ __forceinline__ void mma_bf16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// A chain of NK MMAs accumulating over K steps.  Descriptors advance by compile-time steps in
// 16-byte units (K-major 16-element step: 2; MN-major 16-row step: 128), so issuing one MMA costs
// a few instructions; acc_first says whether the first MMA adds to D.
template <int NK, int ASTEP, int BSTEP>
__device__ __forceinline__ void mma_chain(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t acc_first) {
#pragma unroll
    for (int j = 0; j < NK; ++j)
        mma_bf16(d_tmem, adesc + (uint64_t)(j * ASTEP), bdesc + (uint64_t)(j * BSTEP), idesc, j ? 1u : acc_first);
}
// The same with A in TMEM (8 columns per 16-element K step).
template <int NK, int BSTEP>
__device__ __forceinline__ void mma_chain_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t acc_first) {
#pragma unroll
    for (int j = 0; j < NK; ++j)
        mma_bf16_ta(d_tmem, a_tmem + 8u * j, bdesc + (uint64_t)(j * BSTEP), idesc, j ? 1u : acc_first);
}

// Packs 32 fp32 values (pairs along K) into hi / lo bf16 pair words.
__device__ __forceinline__ void split_pack32(const float *x, uint32_t (&hi)[32], uint32_t (&lo)[32]) {
#pragma unroll
    for (int i = 0; i < 32; ++i) split_pair(x[2 * i], x[2 * i + 1], hi[i], lo[i]);
}
// Packs 16 fp32 values (pairs along K) into hi / lo bf16 pair words.
__device__ __forceinline__ void split_pack16(const float *x, uint32_t (&hi)[16], uint32_t (&lo)[16]) {
#pragma unroll
    for (int i = 0; i < 16; ++i) split_pair(x[2 * i], x[2 * i + 1], hi[i], lo[i]);
}

// 16 consecutive floats of shared memory (16-byte aligned) as four 16-byte loads.
__device__ __forceinline__ void lds16f(const float *src, float (&x)[16]) {
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float4 w = s4[q];
        x[4 * q] = w.x;
        x[4 * q + 1] = w.y;
        x[4 * q + 2] = w.z;
        x[4 * q + 3] = w.w;
    }
}

// 8 consecutive floats of shared memory (16-byte aligned) as two 16-byte loads.
__device__ __forceinline__ void lds8f(const float *src, float (&x)[8]) {
    const float4 a = reinterpret_cast<const float4 *>(src)[0], b = reinterpret_cast<const float4 *>(src)[1];
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

// ------------------------------------------------------------------ swizzled tiles
// A K-major operand tile is stored as blocks of 64 bf16 along K; inside a
// block, row r occupies 128 bytes at r * 128 and its 16-byte chunk c sits at
// chunk position c ^ (r & 7) (the TMA / UMMA 128-byte swizzle).
__device__ __forceinline__ uint32_t sw128_addr(uint32_t block_base, int row, int chunk) {
    return block_base + (uint32_t)row * 128u + ((uint32_t)(chunk ^ (row & 7)) << 4);
}
__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}
__device__ __forceinline__ uint32_t pack_bf16(float lo_elem, float hi_elem) {
    __nv_bfloat162 t = __floats2bfloat162_rn(lo_elem, hi_elem);
    return *reinterpret_cast<uint32_t *>(&t);
}
// The pair (x0, x1) as a hi word {bf16(x0), bf16(x1)} and a lo word {bf16(x0 - hi0), bf16(x1 - hi1)}
// (x0 in the low half of each word): x ~= hi + lo to about 16 significant bits.  One paired
// conversion gives both hi values, which are read back from the word for the residuals.
__device__ __forceinline__ void split_pair(float x0, float x1, uint32_t &hi, uint32_t &lo) {
    hi = pack_bf16(x0, x1);
    lo = pack_bf16(x0 - __uint_as_float(hi << 16), x1 - __uint_as_float(hi & 0xFFFF0000u));
}
// Writes 8 consecutive K elements of one row as hi and lo bf16 chunks.
__device__ __forceinline__ void st_split_chunk(uint32_t hi_block, uint32_t lo_block, int row, int chunk,
                                               const float *x) {
    uint32_t h[4], l[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) split_pair(x[2 * i], x[2 * i + 1], h[i], l[i]);
    st_shared_v4(sw128_addr(hi_block, row, chunk), h[0], h[1], h[2], h[3]);
    st_shared_v4(sw128_addr(lo_block, row, chunk), l[0], l[1], l[2], l[3]);
}

}  // namespace tc
}  // namespace gdn
