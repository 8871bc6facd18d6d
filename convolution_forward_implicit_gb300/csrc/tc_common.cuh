// Device helpers shared by the tensor-core convolution kernels: PTX wrappers for mbarrier,
// TMA/bulk copies and tcgen05, the shared-memory matrix descriptor, the GELU forms, output
// tile decoding and the staged, coalesced epilogue.  Included inside each kernel file.
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

#include "gelu.cuh"
#include "internal.h"

namespace convfwd {
namespace {

constexpr int BM = 128;
constexpr int EPI_WARPS = 8;                           // two per TMEM lane quarter, splitting the columns
constexpr int LAG = 2;                                 // K blocks a cp.async producer keeps in flight
constexpr uint32_t A_BYTES = BM * 128;                 // 128 pixels x 64 bf16
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ unsigned long long globaltimer() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ---- mbarrier ----
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
// try_wait with a suspend-time hint: a waiting thread sleeps until the phase completes (or
// the hint runs out) instead of spinning, so waiting warps do not take issue slots from the
// warps that work.
// Which roles sleep is a plan choice (TcParams::sleep_mask): waking a suspended thread costs
// latency, which matters on the critical path (the MMA issuer, refills of a short ring).
constexpr uint32_t SUSPEND_HINT_NS = 1000000;
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(SUSPEND_HINT_NS)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
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

// Bounded wait.  Returns false if this CTA is aborting (the limit ran out here or elsewhere).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag, unsigned* err,
                                         bool sleep = false) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (sleep ? mbar_try_wait_sleep(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if (globaltimer() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            atomicOr(err, ERR_WAIT_TIMEOUT);
            return false;
        }
    }
}

// Bounded wait taken by lane 0 for the whole (converged) warp; every lane returns lane 0's
// outcome, so a warp never splits at an abort and later meets itself at a warp barrier.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                              unsigned* err, bool sleep = false) {
    int ok = 1;
    if ((threadIdx.x & 31) == 0) ok = wait_bar(bar, parity, abort_flag, err, sleep) ? 1 : 0;
    return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

// ---- async copies ----
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Tiled TMA load of a 5-D box (coordinates innermost first; out-of-range elements read 0).
__device__ __forceinline__ void tma_load_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            int c4, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
        "%5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar)
        : "memory");
}
// L2 prefetch of the same 5-D box (no shared memory, no barrier).  It may run before the
// previous kernel on the stream has completed: it only brings lines into L2, where that kernel's
// writes land as well, so the load issued after griddepcontrol.wait reads current data.
__device__ __forceinline__ void tma_prefetch_5d(const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4) {
    asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
                 : "memory");
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
// The same copy written to every CTA of the cluster in `mask`, at the same shared-memory offset
// in each, completing `bytes` of transaction count on the mbarrier at offset `bar` in each.
__device__ __forceinline__ void bulk_g2s_multicast(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar,
                                                   uint16_t mask) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster [%0], [%1], %2, [%3], "
        "%4;" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar), "h"(mask)
        : "memory");
}

// Tiled TMA store of a 5-D box from shared memory (elements outside the tensor are not
// written), tracked by the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_store_5d(const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4, uint32_t src) {
    asm volatile(
        "cp.async.bulk.tensor.5d.global.shared::cta.bulk_group [%0, {%1, %2, %3, %4, %5}], [%6];" ::"l"(
            reinterpret_cast<uint64_t>(map)),
        "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(src)
        : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the shared-memory sources of this thread's bulk stores have been read (they may be rewritten)
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// this thread's bulk stores have completed
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// ---- tcgen05 ----
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
// Arrive once on the mbarrier at offset `bar` in every CTA of the cluster in `mask` when the
// MMAs issued so far have completed.
__device__ __forceinline__ void mma_commit_multicast(uint32_t bar, uint16_t mask) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"(mask)
        : "memory");
}
// Whole-warp forms: every lane runs the MMA role's loop with the same (warp-uniform)
// descriptors and elect.sync picks the one lane that issues.  In a converged warp it is the
// same lane every time, so the commits below track that lane's MMAs.  Keeping the loop
// uniform, rather than running it in lane 0 alone, lets the descriptor arithmetic stay
// uniform: measured on 128x64 tiles, the issue cost fell from about 70 cycles per MMA.
__device__ __forceinline__ void mma_bf16_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_tf32_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// The four K=16 steps of one 128-byte K block (64 bf16) in one go, issued by the calling
// thread: descriptors advance by 32 bytes (2 in the start-address field) per step; the first
// step accumulates only if `accumulate`, the others always.  (Measured: faster than four
// separate issues in the per-tap kernel; in the slab kernel's whole-warp form, slower on the 2D
// grouped configs.)
__device__ __forceinline__ void mma_bf16_k4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
        "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
        "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %3, t;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %3, t;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void mma_commit_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}
// 32 lanes x 32 bits, 16 consecutive columns: thread t of the warp gets lane (base + t).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}
// 32 lanes x 32 bits, 32 consecutive columns.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
          "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
          "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
        : "r"(taddr));
}
template <int QW>
__device__ __forceinline__ void tmem_ld(uint32_t taddr, uint32_t (&v)[QW]) {
    if constexpr (QW == 32) tmem_ld32(taddr, v);
    else tmem_ld16(taddr, v);
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of 128 B,
// 8-row groups 1024 B apart.  Fields: start address >> 4 (bits 0-13), leading byte
// offset >> 4 (16-29, unused for this layout), stride byte offset >> 4 (32-45),
// descriptor version 1 (46-48), swizzle mode 2 = 128 B (61-63).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction descriptor: D fp32 (bit 4), A and B format (bits 7-9, 10-12: 1 = bf16
// for kind::f16, 2 = tf32 for kind::tf32), both K-major, N >> 3 at bits 17-22, M >> 4 at
// bits 24-28.
__host__ __device__ constexpr uint32_t idesc_f32acc(int m, int n, uint32_t ab_format) {
    return (1u << 4) | (ab_format << 7) | (ab_format << 10) | ((uint32_t)(n >> 3) << 17) |
           ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

// Place in y of GEMM row m (pixels in N Do Ho Wo order) of a lattice-output problem.
__device__ __forceinline__ int out_pixel_linear(const TcParams& p, int m) {
    const int q1 = fdiv(m, p.f_Wo);
    const int ow = m - q1 * p.g.Wo;
    const int q2 = fdiv(q1, p.f_Ho);
    const int oh = q1 - q2 * p.g.Ho;
    const int n = fdiv(q2, p.f_Do);
    const int od = q2 - n * p.g.Do;
    return lattice_pixel(p.lat, n, od, oh, ow);
}

__device__ __forceinline__ void decode_unit(const TcParams& p, int u, int& mt, int& g, int& nt, int& split) {
    const int r = fdiv(u, p.f_splits);
    split = u - r * p.splits;
    const int r2 = fdiv(r, p.f_num_nt);
    nt = r - r2 * p.num_nt;
    mt = fdiv(r2, p.f_G);
    g = r2 - mt * p.g.G;
}

// ---- thread-block clusters ----
// Every thread of every CTA in the cluster arrives; the wait returns once all have (release /
// acquire: shared-memory writes before the arrive are visible to the cluster after the wait).
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// The address of this CTA's shared-memory location saddr in the CTA of cluster rank `rank`.
__device__ __forceinline__ uint32_t cluster_map(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}

// Position in a ring of n pipeline stages: the stage and the parity of its current phase,
// advanced together (no division per step).
struct Ring {
    int n, s;
    uint32_t ph;
    __device__ __forceinline__ explicit Ring(int stages) : n(stages), s(0), ph(0) {}
    __device__ __forceinline__ void next() {
        if (++s == n) {
            s = 0;
            ph ^= 1u;
        }
    }
};

// TMA tiles: mt -> (n, od, oh0, ow0) of a BH x BW block of one output plane.
struct TileOrigin {
    int n, od, oh0, ow0;
};
__device__ __forceinline__ TileOrigin tile_origin(const TcParams& p, int mt) {
    TileOrigin t;
    const int r = fdiv(mt, p.f_tiles_w);
    const int tw = mt - r * p.tiles_w;
    const int r2 = fdiv(r, p.f_tiles_h);
    const int th = r - r2 * p.tiles_h;
    t.n = fdiv(r2, p.f_Do);
    t.od = r2 - t.n * p.g.Do;
    t.oh0 = th * p.BH;
    t.ow0 = tw * p.BW;
    return t;
}

constexpr int STG_WARP_BYTES = 32 * 128;   // one warp's staging buffer: 32 rows x 128 B

// Epilogue of one warp's 32 rows x [cb_begin, cb_end) accumulator columns (see the
// epilogue role in the kernel).  ESZ is the stored element size: 2 for bf16 outputs, 4 for
// fp32 outputs and for split-K partial sums.
// Epilogue geometry of one warp that owns COLS accumulator columns of its 32 rows.
template <int COLS, int ESZ>
struct EpiShape {
    static constexpr int CW = COLS < 128 / ESZ ? COLS : 128 / ESZ;   // columns per chunk
    static constexpr int RB = CW * ESZ;                             // bytes per row segment (32..128)
    static constexpr int LPR = RB / 16;                             // 16-byte slots (= store lanes) per row
    static constexpr int RPI = 32 / LPR;                            // rows per store instruction
};
constexpr int EPI_MAX_LPR = 8;
// Staging bytes one warp's epilogue uses: 32 rows of one chunk's row segments.
template <int COLS, int ESZ>
__host__ __device__ constexpr uint32_t stg_warp_bytes() {
    return 32u * (uint32_t)EpiShape<COLS, ESZ>::RB;
}
// The same on the host side for the slab kernels (BN/2 columns a warp, at least 16).
inline size_t slab_stg_warp_bytes(int BN, int esz) {
    const int cols = BN / 2 < 16 ? 16 : BN / 2;
    const int cw = cols < 128 / esz ? cols : 128 / esz;
    return (size_t)32 * cw * esz;
}

// The output offsets of the rows this lane stores (the same for every chunk of a tile), or -1
// for rows outside the output.  Callers compute them before they wait for the accumulator:
// the index arithmetic (divisions by the tile's extents) then overlaps the MMAs instead of
// delaying the epilogue; the empty asm makes the values exist at that point.
template <int COLS, int ESZ, typename RowOffset>
__device__ __forceinline__ void epilogue_rows(int lane, int wq, RowOffset row_offset, long long (&roff)[EPI_MAX_LPR]) {
    using S = EpiShape<COLS, ESZ>;
#pragma unroll
    for (int i = 0; i < S::LPR; ++i) {
        roff[i] = row_offset(wq * 32 + lane / S::LPR + S::RPI * i);
        asm volatile("" ::"l"(roff[i]));
    }
}

// Where a warp's 32 rows go when the epilogue stores through a tensor map of y: rows are the
// 32 consecutive output pixels starting at (n, od, oh, ow) along W.
struct YBox {
    int ow, oh, od, n;
};

// One warp's share of a tile's epilogue: its 32 accumulator rows (TMEM lane quarter wq) and
// the columns [cb_begin, cb_end) of the BN-wide tile, in chunks of up to COLS columns.  QW32:
// read TMEM 32 columns at a time where the chunk allows (fewer round trips, more registers).
// With ymap (bf16 outputs in 64- or 32-column chunks), each chunk leaves the staging buffer as
// one TMA store of a 64- or 32-channel x 32-pixel box at ybox instead of per-lane stores.
template <int BN, int COLS, int ESZ, bool QW32 = true>
__device__ __forceinline__ void epilogue_chunks(const TcParams& p, uint32_t taddr, int lane, int wq, int cb_begin,
                                                int cb_end, int nt, int gi, int split, bool partial, bool add_bias,
                                                bool do_gelu, uint8_t* stg, const long long (&roff)[EPI_MAX_LPR],
                                                const float* bsm = nullptr, const CUtensorMap* ymap = nullptr,
                                                YBox ybox = YBox{0, 0, 0, 0}) {
    using S = EpiShape<COLS, ESZ>;
    constexpr int CW = S::CW;
    constexpr int RB = S::RB;
    constexpr int LPR = S::LPR;
    constexpr int RPI = S::RPI;
    constexpr int SH = LPR == 8 ? 0 : LPR == 4 ? 1 : LPR == 2 ? 2 : 3;   // log2(8 / LPR)
    constexpr int EPS = 16 / ESZ;                            // elements per 16-byte slot
    const Geom& g = p.g;
    const int GK = g.G * g.K;
    const int slot = lane % LPR;
    const int swz = (lane >> SH) & (LPR - 1);   // this lane's row: slot j sits at j ^ swz
    for (int cb = cb_begin; cb < cb_end; cb += CW) {
        const int n0 = nt * BN + cb;
        if (n0 >= g.K) break;                               // warp-uniform
        if (ESZ == 2 && (CW == 64 || CW == 32) && ymap) {
            // the staging buffer is rewritten only after the previous chunk's store has read it
            if (lane == 0) bulk_wait_read_all();
            __syncwarp();
        }
        // QW columns per TMEM load (32 where the chunk allows): TMEM -> fp32 -> bias, GELU ->
        // this lane's row slots in staging
        // (fp32 outputs keep 16: the 3xTF32 kernels run 544 threads and have fewer registers)
        constexpr int QW = (QW32 && ESZ == 2 && CW % 32 == 0) ? 32 : 16;
#pragma unroll
        for (int q = 0; q < CW / QW; ++q) {
            const int nq = n0 + QW * q;
            // bf16 bias: its loads go out before the TMEM load, so that their latencies overlap
            // (8-column groups past K read as zeros; those columns are never stored)
            uint4 bq[ESZ == 2 ? QW / 8 : 1];
            if (ESZ == 2 && add_bias && !bsm) {
#pragma unroll
                for (int j = 0; j < QW / 8; ++j)
                    bq[j] = nq + 8 * j < g.K ? __ldg(reinterpret_cast<const uint4*>(
                                                         reinterpret_cast<const __nv_bfloat16*>(p.bias) +
                                                         (size_t)gi * g.K + nq) + j)
                                             : make_uint4(0u, 0u, 0u, 0u);
            }
            uint32_t v[QW];
            __syncwarp();                                   // tcgen05.ld is warp-aligned
            tmem_ld<QW>(taddr + (uint32_t)(cb + QW * q), v);
            tmem_ld_wait();
            float f[QW];
#pragma unroll
            for (int e = 0; e < QW; ++e) f[e] = __uint_as_float(v[e]);
            if (ESZ == 2 && add_bias && bsm) {
                // the warp's bias columns, already fp32 in shared memory (one broadcast read per
                // 4 columns)
                const float4* bp = reinterpret_cast<const float4*>(bsm + (cb - cb_begin) + QW * q);
#pragma unroll
                for (int j = 0; j < QW / 4; ++j) {
                    const float4 b = bp[j];
                    add2(f[4 * j], f[4 * j + 1], b.x, b.y);
                    add2(f[4 * j + 2], f[4 * j + 3], b.z, b.w);
                }
            } else if (ESZ == 2 && add_bias) {
#pragma unroll
                for (int j = 0; j < QW / 8; ++j) {
                    const uint32_t bw[4] = {bq[j].x, bq[j].y, bq[j].z, bq[j].w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        add2(f[8 * j + 2 * e], f[8 * j + 2 * e + 1], __uint_as_float(bw[e] << 16),
                             __uint_as_float(bw[e] & 0xFFFF0000u));
                }
            } else if (add_bias) {
                // fp32 bias: only whole 4-column groups inside K are read; columns past K are
                // never stored
#pragma unroll
                for (int j = 0; j < QW / 8; ++j) {
                    if (nq + 8 * j >= g.K) break;
                    const float4* bp =
                        reinterpret_cast<const float4*>(reinterpret_cast<const float*>(p.bias) + (size_t)gi * g.K + nq) +
                        2 * j;
                    const float4 a = __ldg(bp);
                    const float4 b = (nq + 8 * j + 4 < g.K) ? __ldg(bp + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                    add2(f[8 * j], f[8 * j + 1], a.x, a.y);
                    add2(f[8 * j + 2], f[8 * j + 3], a.z, a.w);
                    add2(f[8 * j + 4], f[8 * j + 5], b.x, b.y);
                    add2(f[8 * j + 6], f[8 * j + 7], b.z, b.w);
                }
            }
            if (do_gelu) {
                if (ESZ == 2) {
#pragma unroll
                    for (int e = 0; e < QW; e += 2) gelu2(f[e], f[e + 1]);
                } else {
#pragma unroll
                    for (int e = 0; e < QW; ++e) f[e] = gelu(f[e]);
                }
            }
            constexpr int SPQ = QW / EPS;                   // 16-byte slots per QW columns
#pragma unroll
            for (int t = 0; t < SPQ; ++t) {
                const int j = q * SPQ + t;
                uint4 o;
                if (ESZ == 4) {
                    o = make_uint4(__float_as_uint(f[4 * t]), __float_as_uint(f[4 * t + 1]),
                                   __float_as_uint(f[4 * t + 2]), __float_as_uint(f[4 * t + 3]));
                } else {
                    o.x = pack_bf16x2(f[8 * t + 0], f[8 * t + 1]);
                    o.y = pack_bf16x2(f[8 * t + 2], f[8 * t + 3]);
                    o.z = pack_bf16x2(f[8 * t + 4], f[8 * t + 5]);
                    o.w = pack_bf16x2(f[8 * t + 6], f[8 * t + 7]);
                }
                *reinterpret_cast<uint4*>(stg + lane * RB + ((j ^ swz) << 4)) = o;
            }
        }
        __syncwarp();
        if (ESZ == 2 && (CW == 64 || CW == 32) && ymap) {
            // 32 rows x 128 (64) bytes in the 128-byte (64-byte) swizzle the tensor map expects:
            // one box store
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                tma_store_5d(ymap, gi * g.K + n0, ybox.ow, ybox.oh, ybox.od, ybox.n, smem_u32(stg));
                bulk_commit_group();
            }
            continue;
        }
        // row-wise store: lanes slot..slot+LPR-1 of a row write its whole segment
        const int col = n0 + slot * EPS;
        uint8_t* base = partial ? reinterpret_cast<uint8_t*>(p.ws) + ((size_t)split * g.M * GK) * 4
                                : reinterpret_cast<uint8_t*>(p.y);
#pragma unroll
        for (int i = 0; i < LPR; ++i) {
            const int rr = lane / LPR + RPI * i;           // row within the warp's 32
            const uint4 o = *reinterpret_cast<const uint4*>(stg + rr * RB + ((slot ^ ((rr >> SH) & (LPR - 1))) << 4));
            if (roff[i] >= 0 && col < g.K)
                *reinterpret_cast<uint4*>(base + (size_t)(roff[i] + (long long)gi * g.K + col) * ESZ) = o;
        }
        __syncwarp();                                       // staging is rewritten by the next chunk
    }
}

}  // namespace
}  // namespace convfwd
