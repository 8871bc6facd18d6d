// Implicit-GEMM convolution forward on the sm_103a tensor cores (tcgen05), bf16 in,
// fp32 accumulate in tensor memory, fused bias + GELU epilogue.
//
// GEMM view per group g (page "composable_kernel ... LEARNINGS_GROUPED_CONV.md",
// introduction: NHWGC x GKYXC -> NHWGK): rows m are output pixels (n, od, oh, ow),
// columns are output channels k, and the reduction runs over (tap, c) with c innermost,
// so that one 16-byte chunk of the reduction is 8 consecutive channels of one input
// pixel.  The im2col matrix of page "[ET-VK] conv1d runs at ~3% ...", section "The
// conv2d path already solves this", is never materialised: each A tile is gathered
// straight from the channels-last input, zero-filled where a tap falls in the padding.
//
// One persistent CTA per SM, 9 warps in three roles:
//   warps 0-3  epilogue: tcgen05.ld the 128 x BN accumulator (warp w owns TMEM lanes
//              32w..32w+31), add bias, GELU, round to bf16, 16-byte stores; or store
//              fp32 partials when the reduction is split.
//   warps 4-7  producer: per 64-wide K block, 8 cp.async (16 B, zero-fill) per thread
//              gather the 128 x 128 B activation tile into the 128-byte-swizzled K-major
//              layout; one thread bulk-copies the prepacked weight tile (already in
//              swizzled order) with cp.async.bulk and an mbarrier transaction count.
//   warp 8     MMA: one thread issues tcgen05.mma (M = 128, N = BN, K = 16) x 4 per
//              K block and tcgen05.commit to free the stage; the accumulator is double
//              buffered in TMEM so the epilogue of tile i overlaps the main loop of i+1.
// Every mbarrier wait is bounded: after ~1 s it raises the device error word, sets a
// CTA-wide abort flag and the CTA winds down (drains copies, waits for issued MMAs,
// frees TMEM).
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"

namespace convfwd {
namespace {

constexpr int BM = 128;
constexpr int EPI_WARPS = 4;
constexpr int PROD_WARPS = 4;
constexpr int MMA_WARP = EPI_WARPS + PROD_WARPS;      // warp 8
constexpr int THREADS = (EPI_WARPS + PROD_WARPS + 1) * 32;
constexpr int PROD_THREADS = PROD_WARPS * 32;
constexpr int LAG = 2;                                 // K blocks a producer keeps in flight
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
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                         unsigned* err) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer();
    for (uint32_t n = 1;; ++n) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*abort_flag) return false;
        if ((n & 63u) == 0 && globaltimer() - t0 > WAIT_LIMIT_NS) {
            *abort_flag = 1;
            atomicOr(err, ERR_WAIT_TIMEOUT);
            return false;
        }
    }
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
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

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
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
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
// Instruction descriptor, kind::f16: D fp32 (bit 4), A bf16 (bits 7-9 = 1), B bf16
// (bits 10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16(int m, int n) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ float gelu_f(float v) { return 0.5f * v * (1.0f + erff(v * 0.70710678118654752f)); }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
}

template <int BN>
struct Cfg {
    static constexpr uint32_t B_BYTES = BN * 128;
    static constexpr uint32_t TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;    // power of two for BN in {16..256}
};

__device__ __forceinline__ void decode_unit(const TcParams& p, int u, int& mt, int& g, int& nt, int& split) {
    split = u % p.splits;
    int r = u / p.splits;
    nt = r % p.num_nt;
    r /= p.num_nt;
    g = r % p.g.G;
    mt = r / p.g.G;
}

template <int BN, int STAGES>
__global__ void __launch_bounds__(THREADS, 1) conv_fwd_tc_kernel(const __grid_constant__ TcParams p) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const uint32_t sA = sbase;
    const uint32_t sB = sbase + STAGES * A_BYTES;
    const uint32_t bar0 = sbase + STAGES * (A_BYTES + C::B_BYTES);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    uint8_t* misc = smem + (bar0 + 8u * (2 * STAGES + 5) - sbase);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), PROD_THREADS + 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EPI_WARPS);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const Geom& g = p.g;
    const int GC = g.G * g.C;
    const int GK = g.G * g.K;

    if (warp >= EPI_WARPS && warp < MMA_WARP) {
        // ------------------------------------------------------------ producer
        const int pt = threadIdx.x - EPI_WARPS * 32;
        const int j = pt & 7;        // 16-byte chunk of the 128-byte row
        const int rb = pt >> 3;      // rows rb, rb+16, ..., rb+112
        const uint32_t swz = (uint32_t)((j ^ (rb & 7)) << 4);
        const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x);
        const uint8_t* wp = reinterpret_cast<const uint8_t*>(p.wpack);
        uint32_t it = 0;
        bool aborted = false;
        for (int u = blockIdx.x; u < p.total_units && !aborted; u += gridDim.x) {
            int mt, gi, nt, split;
            decode_unit(p, u, mt, gi, nt, split);
            const int kb0 = split * p.kbps;
            const int kb1 = min(kb0 + p.kbps, p.nkb);
            int rn[8], rd[8], rh[8], rw[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int m = mt * BM + rb + 16 * i;
                if (m < g.M) {
                    int t = m;
                    const int ow = t % g.Wo; t /= g.Wo;
                    const int oh = t % g.Ho; t /= g.Ho;
                    const int od = t % g.Do;
                    rn[i] = t / g.Do;
                    rd[i] = od * g.sd - g.pd;
                    rh[i] = oh * g.sh - g.ph;
                    rw[i] = ow * g.sw - g.pw;
                } else {
                    rn[i] = -1; rd[i] = 0; rh[i] = 0; rw[i] = 0;
                }
            }
            const __nv_bfloat16* xg = x + (size_t)gi * g.C;
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!wait_bar(empty_bar(s), ph ^ 1u, abort_flag, p.err)) { aborted = true; break; }
                if (pt == 0) {
                    mbar_arrive_expect_tx(full_bar(s), C::B_BYTES);
                    const size_t off = ((size_t)(gi * p.num_nt + nt) * p.nkb + kb) * C::B_BYTES;
                    bulk_g2s(sB + s * C::B_BYTES, wp + off, C::B_BYTES, full_bar(s));
                }
                const int q = kb * 8 + j;
                const bool qok = q < p.nchunks;
                const int tap = qok ? q / p.cpt : 0;
                const int c0 = (q - tap * p.cpt) * 8;
                const int zz = tap / (g.Y * g.X);
                const int rem = tap - zz * g.Y * g.X;
                const int yy = rem / g.X;
                const int xx = rem - yy * g.X;
                const int dz = zz * g.dd, dy = yy * g.dh, dx = xx * g.dw;
                const uint32_t dst0 = sA + s * A_BYTES + swz;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int id = rd[i] + dz, ih = rh[i] + dy, iw = rw[i] + dx;
                    const bool ok = qok && rn[i] >= 0 && (unsigned)id < (unsigned)g.D &&
                                    (unsigned)ih < (unsigned)g.H && (unsigned)iw < (unsigned)g.W;
                    const __nv_bfloat16* src =
                        ok ? xg + ((((size_t)rn[i] * g.D + id) * g.H + ih) * g.W + iw) * GC + c0 : x;
                    cp_async_16(dst0 + (uint32_t)(rb + 16 * i) * 128u, src, ok ? 16u : 0u);
                }
                cp_async_commit();
                if (it >= (uint32_t)LAG) {
                    cp_async_wait<LAG>();
                    fence_proxy_async();
                    mbar_arrive(full_bar((it - LAG) % STAGES));
                }
            }
        }
        cp_async_wait<0>();
        fence_proxy_async();
        if (!aborted) {
            const uint32_t first = it > (uint32_t)LAG ? it - LAG : 0u;
            for (uint32_t k = first; k < it; ++k) mbar_arrive(full_bar(k % STAGES));
        }
    } else if (warp == MMA_WARP) {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_bf16(BM, BN);
            uint32_t it = 0, tile_i = 0;
            bool aborted = false;
            for (int u = blockIdx.x; u < p.total_units && !aborted; u += gridDim.x, ++tile_i) {
                int mt, gi, nt, split;
                decode_unit(p, u, mt, gi, nt, split);
                const int kb0 = split * p.kbps;
                const int kb1 = min(kb0 + p.kbps, p.nkb);
                const int acc = tile_i & 1;
                const uint32_t aph = (tile_i >> 1) & 1u;
                if (!wait_bar(tempty_bar(acc), aph ^ 1u, abort_flag, p.err)) { aborted = true; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_bar(full_bar(s), ph, abort_flag, p.err)) { aborted = true; break; }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(sA + s * A_BYTES);
                    const uint64_t bd = sw128_desc(sB + s * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < 4; ++k)   // 4 x K=16 = 64 bf16 = one 128-byte row; +32 B each
                        mma_bf16(d_tmem, ad + 2u * k, bd + 2u * k, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                    mma_commit(empty_bar(s));
                }
                if (!aborted) mma_commit(tfull_bar(acc));
            }
            if (aborted) {
                // wait (bounded) until every MMA issued so far has completed
                mma_commit(drain_bar);
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {}
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int wq = warp;                 // TMEM lane quarter
        const int r = wq * 32 + lane;        // accumulator row = pixel within the tile
        const __nv_bfloat16* bias = reinterpret_cast<const __nv_bfloat16*>(p.bias);
        __nv_bfloat16* y = reinterpret_cast<__nv_bfloat16*>(p.y);
        const bool add_bias = (p.epi == EPI_BIAS || p.epi == EPI_BIAS_GELU) && p.splits == 1;
        const bool do_gelu = (p.epi == EPI_BIAS_GELU || p.epi == EPI_GELU) && p.splits == 1;
        uint32_t tile_i = 0;
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x, ++tile_i) {
            int mt, gi, nt, split;
            decode_unit(p, u, mt, gi, nt, split);
            const int acc = tile_i & 1;
            const uint32_t aph = (tile_i >> 1) & 1u;
            if (!wait_bar(tfull_bar(acc), aph, abort_flag, p.err)) break;
            tc_fence_after();
            const int m = mt * BM + r;
            const bool row_ok = m < g.M;
            const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll 1
            for (int cb = 0; cb < BN; cb += 16) {
                const int n = nt * BN + cb;
                if (n >= g.K) break;                       // warp-uniform
                uint32_t v[16];
                __syncwarp();                              // tcgen05.ld is warp-aligned
                tmem_ld16(taddr + cb, v);
                tmem_ld_wait();
                if (row_ok) {
                float f[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) f[e] = __uint_as_float(v[e]);
                const int halves = (n + 8 < g.K) ? 2 : 1;
                if (p.splits > 1) {
                    float* dst = p.ws + ((size_t)split * g.M + m) * GK + (size_t)gi * g.K + n;
                    for (int h = 0; h < halves; ++h) {
                        reinterpret_cast<float4*>(dst + 8 * h)[0] =
                            make_float4(f[8 * h], f[8 * h + 1], f[8 * h + 2], f[8 * h + 3]);
                        reinterpret_cast<float4*>(dst + 8 * h)[1] =
                            make_float4(f[8 * h + 4], f[8 * h + 5], f[8 * h + 6], f[8 * h + 7]);
                    }
                } else {
                    if (add_bias) {
                        const uint4* bp = reinterpret_cast<const uint4*>(bias + (size_t)gi * g.K + n);
                        for (int h = 0; h < halves; ++h) {
                            const uint4 b4 = __ldg(bp + h);
                            const uint32_t bw[4] = {b4.x, b4.y, b4.z, b4.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e) {
                                f[8 * h + 2 * e] += __uint_as_float(bw[e] << 16);
                                f[8 * h + 2 * e + 1] += __uint_as_float(bw[e] & 0xFFFF0000u);
                            }
                        }
                    }
                    if (do_gelu) {
#pragma unroll
                        for (int e = 0; e < 16; ++e) f[e] = gelu_f(f[e]);
                    }
                    __nv_bfloat16* dst = y + (size_t)m * GK + (size_t)gi * g.K + n;
                    for (int h = 0; h < halves; ++h) {
                        uint4 o;
                        o.x = pack_bf16x2(f[8 * h + 0], f[8 * h + 1]);
                        o.y = pack_bf16x2(f[8 * h + 2], f[8 * h + 3]);
                        o.z = pack_bf16x2(f[8 * h + 4], f[8 * h + 5]);
                        o.w = pack_bf16x2(f[8 * h + 6], f[8 * h + 7]);
                        reinterpret_cast<uint4*>(dst + 8 * h)[0] = o;
                    }
                }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int STAGES>
constexpr size_t smem_bytes_for() {
    return 1024 + (size_t)STAGES * (A_BYTES + Cfg<BN>::B_BYTES) + 8 * (2 * STAGES + 5) + 16;
}

template <int BN, int STAGES>
cudaError_t launch_one(const TcParams& p, int grid, cudaStream_t stream) {
    auto kern = conv_fwd_tc_kernel<BN, STAGES>;
    constexpr size_t smem = smem_bytes_for<BN, STAGES>();
    static_assert(smem <= 232448, "shared memory budget");
    // opt in to the large dynamic shared memory once per device (not inside graph capture)
    static bool attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    kern<<<grid, THREADS, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

// (BN, stages) pairs compiled into the library; the plan picks one.
#define TC_CONFIGS(X) X(256, 4) X(128, 6) X(64, 8) X(32, 8) X(16, 8)

bool tc_config_supported(int BN, int stages) {
#define X(bn, st) if (BN == bn && stages == st) return true;
    TC_CONFIGS(X)
#undef X
    return false;
}

size_t tc_smem_bytes(int BN, int stages) {
#define X(bn, st) if (BN == bn && stages == st) return smem_bytes_for<bn, st>();
    TC_CONFIGS(X)
#undef X
    return 0;
}

cudaError_t launch_tc_bf16(const TcParams& p, int stages, int grid, cudaStream_t stream) {
#define X(bn, st) if (p.BN == bn && stages == st) return launch_one<bn, st>(p, grid, stream);
    TC_CONFIGS(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace convfwd
