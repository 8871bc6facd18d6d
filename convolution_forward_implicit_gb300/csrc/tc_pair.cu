// Implicit-GEMM convolution forward on CTA pairs (tcgen05 .cta_group::2): the per-tap bf16
// kernel of tc_conv.cu with an M = 256 accumulator split over the two CTAs of a cluster.
//
// Why: in the one-CTA kernel every 128x256 tile's K block moves 48 KB into shared memory (a
// 16 KB activation box and a 32 KB weight tile) and its four 128x256x16 MMAs read 48 KB back
// out, ~96 KB per 512 cycles of math; shared memory passes ~128 B per cycle, so a K block took
// ~750 cycles on the 1280 -> 1280 conv1d (measured at two clock speeds: the bound scales with
// the SM clock, not memory latency).  A CTA pair computes a 256x256 tile with one M = 256
// MMA stream: each CTA holds its own 128 rows of the activation box and one half (BN/2 rows)
// of each weight tile, and the tensor cores of both SMs read the two halves of B from the two
// shared memories.  Per SM and K block that is 32 KB in and 32 KB read, ~64 KB per 512 cycles.
//
// The pair's protocol (measured semantics of the M = 256 MMA: CTA r holds rows 128r.. of A and
// columns (BN/2)r.. of B at the same shared-memory offsets as its peer; its tensor memory holds
// rows 128r.. of D, all BN columns):
//   * both CTAs' producers load their A box and B half with .cta_group::2 TMA copies that
//     complete on the full barrier of the even CTA (the leader), whose producer alone posts
//     the expected byte count of both CTAs' copies;
//   * the leader's MMA thread waits on its full barrier, issues the M = 256 MMAs and commits
//     each stage to the empty barriers of both CTAs (multicast), and each accumulator to both
//     CTAs' accumulator-full barriers;
//   * each CTA's epilogue drains its own 128 rows and arrives on the leader's accumulator-empty
//     barrier (the peer's warps remotely), which counts both CTAs' epilogue warps;
//   * tensor memory is allocated and freed by one warp in each CTA together.
// Every wait is bounded as in the one-CTA kernel; each CTA drains the arrivals the other may
// still send it before the pair meets at a cluster barrier and frees its tensor memory.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "tc_common.cuh"

namespace convfwd {
namespace {

template <int EW>
struct PairTraits {
    static constexpr int PROD_WARPS = EW == 16 ? 3 : 4;   // 20 or 13 warps in all (96 / 152 registers)
    static constexpr int MMA_WARP = EW + PROD_WARPS;
    static constexpr int THREADS = (MMA_WARP + 1) * 32;
};

template <int BN, int STAGES, int EW>
struct PairSmem {
    static constexpr uint32_t A_STAGE = A_BYTES;              // 128 pixels x 128 bytes
    static constexpr uint32_t B_HALF = (BN / 2) * 128;        // this CTA's half of a weight tile
    static constexpr size_t RING = (size_t)STAGES * (A_STAGE + B_HALF);
    static constexpr size_t STG = (size_t)EW * STG_WARP_BYTES;
    static constexpr size_t BARS = 8 * (3 * STAGES + 5) + 16;
    static constexpr size_t TOTAL = 1024 + RING + STG + BARS;
};

// ---- CTA-pair forms of the tcgen05 and TMA operations ----
__device__ __forceinline__ void tmem_alloc_pair(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// The four K = 16 steps of one 128-byte K block, M = 256 over the pair.
__device__ __forceinline__ void mma_pair_k4(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, t;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
        "setp.ne.b32 p, %4, 0;\n\tsetp.eq.b32 t, 0, 0;\n\t"
        "add.s64 a1, %1, 2;\n\tadd.s64 a2, %1, 4;\n\tadd.s64 a3, %1, 6;\n\t"
        "add.s64 b1, %2, 2;\n\tadd.s64 b2, %2, 4;\n\tadd.s64 b3, %2, 6;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], a1, b1, %3, t;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], a2, b2, %3, t;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], a3, b3, %3, t;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the mbarrier at offset `bar` in both CTAs of the pair when the MMAs issued so
// far have completed.
__device__ __forceinline__ void commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
        "h"((uint16_t)0x3)
        : "memory");
}
__device__ __forceinline__ void commit_pair_local(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}
// Tiled TMA loads into this CTA's shared memory that complete on an mbarrier of either CTA of
// the pair (bar_cluster: a shared::cluster address).
__device__ __forceinline__ void tma_load_5d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                                 int c4, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar_cluster)
        : "memory");
}
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                                 uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar_cluster)
        : "memory");
}
// Remote arrival of the odd CTA's epilogue on the leader's accumulator-empty barrier.  Relaxed:
// it only says that this warp's tensor-memory loads have completed (tcgen05.wait::ld), which the
// tcgen05 fence before it orders; a release at cluster scope would also hold the arrival until
// the warp's global stores of y were acknowledged, which delayed every other unit of the 2D
// grouped layers by 1-2 us (clock stamps).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

template <int BN, int STAGES, int EW>
__global__ void __launch_bounds__(PairTraits<EW>::THREADS, 1)
    conv_fwd_pair_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap act_map,
                         const __grid_constant__ CUtensorMap w_map, const __grid_constant__ CUtensorMap y_map) {
    using T = PairTraits<EW>;
    using SM = PairSmem<BN, STAGES, EW>;
    constexpr uint32_t TMEM_COLS = 2 * BN;                   // two accumulators of BN columns
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const uint32_t sA = sbase;
    const uint32_t sB = sbase + STAGES * SM::A_STAGE;
    constexpr uint32_t STG_OFFSET = (uint32_t)SM::RING;
    const uint32_t bar0 = sbase + STG_OFFSET + (uint32_t)SM::STG;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (2 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
    uint8_t* misc = smem + (bar0 + 8u * (3 * STAGES + 5) - sbase);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const bool leader = crank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);        // the leader's producer (both CTAs' bytes)
            mbar_init(empty_bar(s), 1);       // the leader's commit, multicast to both
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), 2 * EW);   // both CTAs' epilogue warps (used in the leader)
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == EW && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&act_map)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&w_map)) : "memory");
    }
    if (warp == T::MMA_WARP) {
        tmem_alloc_pair(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    // barriers of both CTAs exist before either sends the other a copy or an arrival
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (p.pdl) griddep_launch();

    const Geom& g = p.g;
    const int GK = g.G * g.K;
    const int u0 = (int)(blockIdx.x >> 1), ustep = (int)(gridDim.x >> 1);
    auto unit_tile = [&](int u, int& mt, int& gi, int& nt, int& split) {
        decode_unit(p, u, mt, gi, nt, split);
        mt = 2 * mt + (int)crank;
    };

    if (warp >= EW && warp < T::MMA_WARP) {
        // -------------------------------------------------------------- producers (both CTAs)
        const int pw = warp - EW;
        if (lane < 2) {
            const uint32_t a_tx = (uint32_t)(p.BW * p.BH) * 128u;
            const uint32_t full_leader0 = cluster_map(full_bar(0), 0u);   // + 8 s: stage s
            uint32_t it = 0;
            bool aborted = false;
            bool x_ready = !p.pdl;
            if (!x_ready && lane == 0 && u0 < p.total_units) {
                // this warp's activation boxes of the first unit's first stages go into L2 while
                // the previous kernel finishes
                int mt, gi, nt, split;
                unit_tile(u0, mt, gi, nt, split);
                if (mt < p.num_mt) {
                    const TileOrigin to = tile_origin(p, mt);
                    for (int kb = pw; kb < p.nkb && kb < STAGES; kb += T::PROD_WARPS) {
                        const int tap = fdiv(kb, p.f_cbt);
                        const int c0 = (kb - tap * p.cbt) * 64;
                        const int zz = fdiv(tap, p.f_YX);
                        const int rem = tap - zz * g.Y * g.X;
                        const int yy = fdiv(rem, p.f_X);
                        const int xx = rem - yy * g.X;
                        const int wi = to.ow0 * g.sw - g.pw + xx * g.dw, hi = to.oh0 * g.sh - g.ph + yy * g.dh;
                        if (p.map_kind == 0)
                            tma_prefetch_5d(&act_map, gi * g.C + c0, wi, hi, to.od * g.sd - g.pd + zz * g.dd, to.n);
                        else
                            tma_prefetch_5d(&act_map, c0, gi, wi, hi, to.n);
                    }
                }
            }
            for (int u = u0; u < p.total_units && !aborted; u += ustep) {
                int mt, gi, nt, split;
                unit_tile(u, mt, gi, nt, split);
                // (the second tile of the last pair may lie past the output: its boxes read zeros
                // and its epilogue stores nothing)
                const TileOrigin to = tile_origin(p, mt);
                const int w0 = to.ow0 * g.sw - g.pw, h0 = to.oh0 * g.sh - g.ph, d0 = to.od * g.sd - g.pd;
                const int wrow0 = ((gi * p.num_nt + nt) * p.nkb) * BN + (int)crank * (BN / 2);
                for (int kb = 0; kb < p.nkb; ++kb, ++it) {
                    if ((int)((it % STAGES) % T::PROD_WARPS) != pw) continue;
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    int ok = 1;
                    if (lane == 0) ok = wait_bar(empty_bar(s), ph ^ 1u, abort_flag, p.err, p.sleep_mask & 1) ? 1 : 0;
                    ok = __shfl_sync(0x3u, ok, 0);
                    if (!ok) { aborted = true; break; }
                    if (leader && lane == 0) mbar_arrive_expect_tx(full_bar(s), 2u * (a_tx + SM::B_HALF));
                    __syncwarp(0x3u);
                    const uint32_t fb = full_leader0 + 8u * (uint32_t)s;
                    if (lane == 0) {
                        if (!x_ready) {
                            griddep_wait();
                            x_ready = true;
                        }
                        const int tap = fdiv(kb, p.f_cbt);
                        const int c0 = (kb - tap * p.cbt) * 64;
                        const int zz = fdiv(tap, p.f_YX);
                        const int rem = tap - zz * g.Y * g.X;
                        const int yy = fdiv(rem, p.f_X);
                        const int xx = rem - yy * g.X;
                        const int wi = w0 + xx * g.dw, hi = h0 + yy * g.dh;
                        if (p.map_kind == 0)
                            tma_load_5d_pair(sA + s * SM::A_STAGE, &act_map, gi * g.C + c0, wi, hi, d0 + zz * g.dd,
                                             to.n, fb);
                        else
                            tma_load_5d_pair(sA + s * SM::A_STAGE, &act_map, c0, gi, wi, hi, to.n, fb);
                    } else {
                        tma_load_2d_pair(sB + s * SM::B_HALF, &w_map, 0, wrow0 + kb * BN, fb);
                    }
                }
            }
            if (lane == 0) {
                // before this CTA may leave, every commit the leader sends to its empty barriers
                // must have arrived: wait (bounded) for the phases of this warp's next refills
                for (uint32_t k = it; k < it + (uint32_t)STAGES && !aborted; ++k)
                    if ((int)((k % STAGES) % T::PROD_WARPS) == pw &&
                        !wait_bar(empty_bar(k % STAGES), ((k / STAGES) & 1u) ^ 1u, abort_flag, p.err, false))
                        break;
            }
        }
        __syncwarp();
    } else if (warp == T::MMA_WARP) {
        // -------------------------------------------------------------- MMA issue (leader only)
        if (p.pdl) griddep_wait();
        if (leader && lane == 0) {
            constexpr uint32_t IDESC = idesc_f32acc(256, BN, 1u);
            uint32_t it = 0, tile_i = 0;
            bool aborted = false;
            if (p.test_stall && !wait_bar(drain_bar, 0u, abort_flag, p.err, false)) aborted = true;
            for (int u = u0; u < p.total_units && !aborted; u += ustep, ++tile_i) {
                const int acc = tile_i & 1;
                const uint32_t aph = (tile_i >> 1) & 1u;
                if (!wait_bar(tempty_bar(acc), aph ^ 1u, abort_flag, p.err, (p.sleep_mask & 4) != 0)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < p.nkb; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_bar(full_bar(s), ph, abort_flag, p.err, (p.sleep_mask & 4) != 0)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    mma_pair_k4(d_tmem, sw128_desc(sA + s * SM::A_STAGE), sw128_desc(sB + s * SM::B_HALF), IDESC,
                                kb > 0 ? 1u : 0u);
                    commit_pair(empty_bar(s));
                }
                if (!aborted) commit_pair(tfull_bar(acc));
            }
            if (aborted) {
                // wait (bounded) until every MMA issued so far has completed
                commit_pair_local(drain_bar);
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(drain_bar, 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {}
            } else {
                // every epilogue arrival (the peer's are remote) must have landed before the
                // leader leaves: wait (bounded) as if two more tiles were to start
                for (uint32_t t = tile_i; t < tile_i + 2u; ++t)
                    if (!wait_bar(tempty_bar(t & 1), ((t >> 1) & 1u) ^ 1u, abort_flag, p.err, false)) break;
            }
        }
        __syncwarp();
    } else if (warp < EW) {
        // -------------------------------------------------------------- epilogue (both CTAs)
        const int wq = warp & 3;
        constexpr int COLS = BN / (EW / 4);
        const int cb_begin = (warp >> 2) * COLS;
        const int cb_end = cb_begin + COLS < BN ? cb_begin + COLS : BN;
        const bool add_bias = p.epi == EPI_BIAS || p.epi == EPI_BIAS_GELU;
        const bool do_gelu = p.epi == EPI_BIAS_GELU || p.epi == EPI_GELU;
        uint8_t* stg = smem + STG_OFFSET + warp * STG_WARP_BYTES;
        const uint32_t tempty_leader0 = cluster_map(tempty_bar(0), 0u);
        if (p.pdl) griddep_wait();
        uint32_t tile_i = 0;
        for (int u = u0; u < p.total_units; u += ustep, ++tile_i) {
            int mt, gi, nt, split;
            unit_tile(u, mt, gi, nt, split);
            const int acc = tile_i & 1;
            const uint32_t aph = (tile_i >> 1) & 1u;
            const TileOrigin to = tile_origin(p, mt);
            auto row_offset = [&](int rr) -> long long {
                const int rh = fdiv(rr, p.f_BW);
                const int oh = to.oh0 + rh, ow = to.ow0 + (rr - rh * p.BW);
                if (rr >= p.BW * p.BH || oh >= g.Ho || ow >= g.Wo || to.n >= g.N) return -1;
                return (long long)lattice_pixel(p.lat, to.n, to.od, oh, ow) * GK;
            };
            long long roff[EPI_MAX_LPR];
            epilogue_rows<COLS, 2>(lane, wq, row_offset, roff);
            if (!wait_bar_warp(tfull_bar(acc), aph, abort_flag, p.err, (p.sleep_mask & 2) != 0)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * BN);
            epilogue_chunks<BN, COLS, 2, EW == 8>(p, taddr, lane, wq, cb_begin, cb_end, nt, gi, 0, false, add_bias,
                                                  do_gelu, stg, roff, nullptr, p.ystore ? &y_map : nullptr,
                                                  YBox{to.ow0 + wq * 32, to.oh0, to.od, to.n});
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(tempty_bar(acc));
                else mbar_arrive_cluster(tempty_leader0 + 8u * (uint32_t)acc);
            }
        }
        // the tensor-map stores have completed before this CTA may leave
        if (p.ystore && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    // neither CTA leaves while the other may still copy into or arrive on its shared memory
    cluster_sync_all();
    if (warp == T::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, TMEM_COLS);
    }
}

template <int BN, int STAGES, int EW>
cudaError_t launch_pair_one(const TcParams& p, const CUtensorMap& amap, const CUtensorMap& wmap,
                            const CUtensorMap& ymap, int grid, cudaStream_t stream) {
    auto kern = conv_fwd_pair_kernel<BN, STAGES, EW>;
    constexpr size_t smem = PairSmem<BN, STAGES, EW>::TOTAL;
    static_assert(smem <= 232448, "shared memory budget");
    static bool attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    return launch_kernel(kern, dim3(grid), dim3(PairTraits<EW>::THREADS), smem, stream, p.pdl != 0, 2, p, amap, wmap,
                         ymap);
}

}  // namespace

// (BN, stages, epilogue warps) of the pair kernel: 6 / 4 stages of 32 KB with 8 / 16 epilogue
// warps at BN = 256; 8 / 6 stages of 24 KB at BN = 128.
#define TC_PAIR_CONFIGS(X) X(256, 6, 8) X(256, 4, 16) X(128, 8, 8) X(128, 6, 16)

int tc_pair_stages_for(int BN, int epi_warps) {
#define X(bn, st, ew) if (BN == bn && epi_warps == ew) return st;
    TC_PAIR_CONFIGS(X)
#undef X
    return 0;
}

int tc_pair_max_clusters(int BN, int epi_warps) {
    auto query = [&](auto kern, size_t smem, int threads) -> int {
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2);
        cfg.blockDim = dim3(threads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        return n;
    };
#define X(bn, st, ew)                                                                                   \
    if (BN == bn && epi_warps == ew)                                                                    \
        return query(conv_fwd_pair_kernel<bn, st, ew>, PairSmem<bn, st, ew>::TOTAL, PairTraits<ew>::THREADS);
    TC_PAIR_CONFIGS(X)
#undef X
    return 0;
}

cudaError_t launch_pair(const TcParams& p, const CUtensorMap* act_map, const CUtensorMap* w_map,
                        const CUtensorMap* y_map, int stages, int grid, cudaStream_t stream) {
    static const CUtensorMap unused{};
    if (!act_map || !w_map || !p.tma || p.tf32 || p.splits != 1 || p.cluster_red || (grid & 1))
        return cudaErrorInvalidValue;
    if (p.ystore && (!y_map || p.lat.on || p.BH != 1 || p.BW % 32 != 0)) return cudaErrorInvalidValue;
#define X(bn, st, ew)                                                                \
    if (p.BN == bn && stages == st && p.epi_warps == ew)                             \
        return launch_pair_one<bn, st, ew>(p, *act_map, *w_map, y_map ? *y_map : unused, grid, stream);
    TC_PAIR_CONFIGS(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace convfwd
