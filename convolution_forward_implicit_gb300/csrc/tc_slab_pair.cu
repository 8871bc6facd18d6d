// Slab-mode implicit GEMM (tc_slab.cu) on CTA pairs: M = 256 MMAs (tcgen05 .cta_group::2) whose
// 128-row halves come from the two CTAs of a cluster, each with its own slab.
//
// Why: with N = 64 output channels per group, a 128x64x16 MMA cannot run faster than ~48
// cycles (it reads 4 KB of activations and 2 KB of weights from shared memory; measured by a
// standalone probe), and in the slab kernel the slab and weight copies and the epilogue's
// staging share that bandwidth, so an MMA took ~70 cycles.  On a CTA pair each SM keeps its own
// slab but only half of every weight tile (BN/2 rows per tap), and each M = 256 MMA reads a 1 KB
// weight half per SM: per unit of the 3D G=4 C=K=64 layer, shared-memory traffic falls by about
// a fifth, and with resident weights (2D) half the weight space makes room for a third slab stage.
//
// Pair protocol (the per-tap pair kernel's, tc_pair.cu): both CTAs' slab and weight copies
// (.cta_group::2 TMA) complete on the leader's barriers, whose copy warps alone post the byte
// counts of both CTAs; the leader's MMA warps (one per accumulator of a unit) commit
// every release to both CTAs' barriers; both epilogues arrive on the leader's accumulator-empty
// barrier; tensor memory is allocated and freed by both CTAs together.  Every wait is bounded;
// each CTA drains the arrivals the other may still send it before the cluster barrier at exit.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "tc_common.cuh"

namespace convfwd {
namespace {

constexpr int SP_MAX_SA = 4;
constexpr int SP_MAX_SB = 8;
constexpr int SP_A_WARP = EPI_WARPS;          // slab copies
constexpr int SP_B_WARP0 = EPI_WARPS + 1;     // weight copies (3 warps)
constexpr int SP_B_WARPS = 3;
constexpr int SP_MMA_WARP = EPI_WARPS + 4;    // one MMA warp per accumulator (leader only issues; the
                                              // second idles in one-accumulator units)
constexpr int SP_THREADS = (SP_MMA_WARP + 2) * 32;

__device__ __forceinline__ void sp_tmem_alloc(uint32_t slot_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_smem), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void sp_tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void sp_tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// Whole-warp issue of one M = 256 MMA over the pair (elect.sync picks the issuing lane).
__device__ __forceinline__ void sp_mma_warp(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p, e;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on the barrier at offset `bar` in both CTAs when this thread's MMAs have completed.
__device__ __forceinline__ void sp_commit_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::"r"(
            bar),
        "h"((uint16_t)0x3)
        : "memory");
}
__device__ __forceinline__ void sp_commit_local_warp(uint32_t bar) {
    asm volatile(
        "{\n\t.reg .pred e;\n\t"
        "elect.sync _|e, 0xffffffff;\n\t"
        "@e tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void sp_tma_5d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2, int c3, int c4,
                                          uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3, %4, %5, %6}], [%7];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4), "r"(bar_cluster)
        : "memory");
}
// one weight stage of this CTA: its half (BN/2 rows) of each of the stage's consecutive tap tiles
__device__ __forceinline__ void sp_tma_w(uint32_t dst, const CUtensorMap* map, int half, int tap, uint32_t bar_cluster) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3, %4, %5}], [%6];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(half), "r"(tap), "r"(bar_cluster)
        : "memory");
}
// Remote arrival of the odd CTA's epilogue on the leader's accumulator-empty barrier.  Relaxed:
// it only says that this warp's tensor-memory loads have completed (tcgen05.wait::ld), which the
// tcgen05 fence before it orders; a release at cluster scope would also hold the arrival until
// the warp's global stores of y were acknowledged, which delayed every other unit of the 2D
// grouped layers by 1-2 us (clock stamps).
__device__ __forceinline__ void sp_arrive_cluster(uint32_t bar_cluster) {
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// BY, BT: filter rows and columns fixed at compile time (3x3 filters), 0: from the parameters.
// NACC: 128-row accumulators per CTA and unit, stacked along H (2: a tile pair sharing one slab;
// 1: one accumulator per slab, for slabs too tall to leave room for a weight ring), each issued
// by its own MMA warp.  Units are pairs of slab units; the CTA of cluster rank r takes slab unit
// 2 mt + r.
template <int BN, int BY, int BT, int NACC>
__global__ void __launch_bounds__(SP_THREADS, 1)
    conv_fwd_slab_pair_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap act_map,
                              const __grid_constant__ CUtensorMap w_map) {
    constexpr uint32_t B_HALF = (BN / 2) * 128;                 // one tap's half weight tile
    constexpr uint32_t TMEM_COLS = (2 * NACC * BN < 32) ? 32 : 2 * NACC * BN;
    const int SA = p.slab_sa, SB = p.slab_sb;
    const uint32_t a_stage = (uint32_t)p.slab_a_stage;
    const int nbg = BY > 0 ? BY : p.slab_nbg;
    const int btaps = BT > 0 ? BT : p.slab_btaps;
    const uint32_t b_stage = (uint32_t)btaps * B_HALF;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const uint32_t sA = sbase;
    const uint32_t sB = sA + SA * a_stage;
    const uint32_t stg_off = SA * a_stage + SB * b_stage;
    // each epilogue warp stages one chunk of its BN/2 columns: 32 rows x (BN/2 x element size)
    constexpr uint32_t STG_W = stg_warp_bytes<(BN / 2 < 16 ? 16 : BN / 2), (2)>();
    const uint32_t bar0 = sbase + stg_off + EPI_WARPS * STG_W;
    auto full_a = [&](int s) { return bar0 + 8u * s; };
    auto empty_a = [&](int s) { return bar0 + 8u * (SP_MAX_SA + s); };
    auto full_b = [&](int s) { return bar0 + 8u * (2 * SP_MAX_SA + s); };
    auto empty_b = [&](int s) { return bar0 + 8u * (2 * SP_MAX_SA + SP_MAX_SB + s); };
    const uint32_t bar_t = bar0 + 8u * (2 * SP_MAX_SA + 2 * SP_MAX_SB);
    auto tfull_bar = [&](int a) { return bar_t + 8u * a; };
    auto tempty_bar = [&](int a) { return bar_t + 8u * (2 + a); };
    auto drain_bar = [&](int mw) { return bar_t + 8u * (4 + mw); };
    uint8_t* misc = smem + (bar_t + 8u * 6 - sbase);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t crank = cluster_ctarank();
    const bool leader = crank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(full_a(s), 1);          // the leader's slab warp (both CTAs' bytes)
            mbar_init(empty_a(s), NACC);      // the leader's MMA warps, multicast to both
        }
        if (p.slab_resident) {
            mbar_init(full_b(0), SP_B_WARPS);
            mbar_init(empty_b(0), NACC);
        } else {
            for (int s = 0; s < SB; ++s) {
                mbar_init(full_b(s), 1);
                mbar_init(empty_b(s), NACC);
            }
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), NACC);
            mbar_init(tempty_bar(a), 2 * EPI_WARPS);   // both CTAs' epilogue warps (used in the leader)
        }
        for (int mw = 0; mw < NACC; ++mw) mbar_init(drain_bar(mw), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == SP_A_WARP && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&act_map)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&w_map)) : "memory");
    }
    if (warp == SP_MMA_WARP) {
        sp_tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        sp_tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    if (p.pdl) griddep_launch();

    const Geom& g = p.g;
    const int u0 = (int)(blockIdx.x >> 1), ustep = (int)(gridDim.x >> 1);
    auto unit_tile = [&](int u, int& mt, int& gi, int& nt) {
        int split;
        decode_unit(p, u, mt, gi, nt, split);
        mt = 2 * mt + (int)crank;
    };

    if (warp == SP_A_WARP) {
        // ------------------------------------------------------------ slab copies (both CTAs)
        if (lane == 0) {
            if (p.pdl) griddep_wait();
            const uint32_t a_tx = (uint32_t)(p.slab_hr * p.slab_bws) * 128u;
            const uint32_t full_leader0 = cluster_map(full_a(0), 0u);
            Ring ra(SA);
            uint32_t it = 0;
            bool aborted = false;
            for (int u = u0; u < p.total_units && !aborted; u += ustep) {
                int mt, gi, nt;
                unit_tile(u, mt, gi, nt);
                // (the second slab unit of the last pair may lie past the output: its box reads zeros)
                const TileOrigin to = tile_origin(p, mt);
                const int w0 = to.ow0 - g.pw, h0 = to.oh0 - g.ph;
                for (int kg = 0; kg < p.slab_nkg; ++kg, ra.next(), ++it) {
                    const int zz = fdiv(kg, p.f_cbt), cb = kg - zz * p.cbt;
                    const int s = ra.s;
                    if (!wait_bar(empty_a(s), ra.ph ^ 1u, abort_flag, p.err, p.sleep_mask & 1)) { aborted = true; break; }
                    if (leader) mbar_arrive_expect_tx(full_a(s), 2u * a_tx);
                    const uint32_t fb = full_leader0 + 8u * (uint32_t)s;
                    if (p.map_kind == 0)
                        sp_tma_5d(sA + s * a_stage, &act_map, gi * g.C + cb * 64, w0, h0, to.od - g.pd + zz * g.dd,
                                  to.n, fb);
                    else
                        sp_tma_5d(sA + s * a_stage, &act_map, cb * 64, gi, w0, h0, to.n, fb);
                }
            }
            // every release the leader commits to this CTA's slab stages has arrived before exit
            for (uint32_t k = it; k < it + (uint32_t)SA && !aborted; ++k)
                if (!wait_bar(empty_a(k % SA), ((k / SA) & 1u) ^ 1u, abort_flag, p.err, false)) break;
        }
        __syncwarp();
    } else if (warp >= SP_B_WARP0 && warp < SP_B_WARP0 + SP_B_WARPS) {
        // ------------------------------------------------------------ weight copies (both CTAs)
        if (lane == 0) {
            const int bw = warp - SP_B_WARP0;
            const int nchunk = p.slab_nkg * nbg;     // chunks of btaps taps, in slab order
            bool aborted = false;
            if (p.slab_resident) {
                // the weight set of the current (group, N tile), this CTA's half of every tap
                const uint32_t fb = cluster_map(full_b(0), 0u);
                int prev = -1;
                uint32_t j = 0;
                for (int u = u0; u < p.total_units && !aborted; u += ustep) {
                    int mt, gi, nt;
                    unit_tile(u, mt, gi, nt);
                    const int key = gi * p.num_nt + nt;
                    if (key == prev) continue;
                    prev = key;
                    if (p.pdl && j == 1) griddep_wait();
                    if (!wait_bar(empty_b(0), (j & 1u) ^ 1u, abort_flag, p.err, p.sleep_mask & 1)) {
                        aborted = true;
                        break;
                    }
                    const int mine = nchunk > bw ? (nchunk - bw + SP_B_WARPS - 1) / SP_B_WARPS : 0;
                    if (leader) mbar_arrive_expect_tx(full_b(0), 2u * (uint32_t)mine * b_stage);
                    for (int c = bw; c < nchunk; c += SP_B_WARPS)
                        sp_tma_w(sB + c * b_stage, &w_map, (int)crank, key * p.nkb + c * btaps, fb);
                    ++j;
                }
                // the leader's release of the last weight set has arrived before exit
                if (!aborted) wait_bar(empty_b(0), (j & 1u) ^ 1u, abort_flag, p.err, false);
            } else {
                const uint32_t fb0 = cluster_map(full_b(0), 0u);
                uint32_t ib = 0;
                Ring rb(SB);
                bool waited = false;
                for (int u = u0; u < p.total_units && !aborted; u += ustep) {
                    int mt, gi, nt;
                    unit_tile(u, mt, gi, nt);
                    const int tap0 = (gi * p.num_nt + nt) * p.nkb;
                    for (int c = 0; c < nchunk; ++c, ++ib, rb.next()) {
                        const int s = rb.s;
                        if (s % SP_B_WARPS != bw) continue;
                        if (p.pdl && ib >= (uint32_t)SB && !waited) {
                            griddep_wait();
                            waited = true;
                        }
                        if (!wait_bar(empty_b(s), rb.ph ^ 1u, abort_flag, p.err, p.sleep_mask & 1)) {
                            aborted = true;
                            break;
                        }
                        if (leader) mbar_arrive_expect_tx(full_b(s), 2u * b_stage);
                        sp_tma_w(sB + s * b_stage, &w_map, (int)crank, tap0 + c * btaps, fb0 + 8u * (uint32_t)s);
                    }
                }
                // every release of this warp's stages has arrived before exit
                for (uint32_t k = ib; k < ib + (uint32_t)SB && !aborted; ++k)
                    if ((int)((k % SB) % SP_B_WARPS) == bw &&
                        !wait_bar(empty_b(k % SB), ((k / SB) & 1u) ^ 1u, abort_flag, p.err, false))
                        break;
            }
        }
        __syncwarp();
    } else if (warp >= SP_MMA_WARP && warp < SP_MMA_WARP + NACC) {
        // ------------------------------------------------------------ MMA issue (leader only)
        // warp mw issues accumulator mw of every unit; both wait for the same stages
        const int mw = warp - SP_MMA_WARP;
        if (p.pdl) griddep_wait();
        if (leader) {
            constexpr uint32_t IDESC = idesc_f32acc(256, BN, 1u);
            const bool msleep = (p.sleep_mask & 4) != 0;
            const bool resident = p.slab_resident != 0;
            const int KT = p.g.G * p.num_nt;
            const int kstep = ustep % KT;
            int key = u0 % KT;
            Ring ra(SA), rb(SB);
            uint32_t tile_i = 0, jw = 0;
            int prev = -1;
            bool aborted = false;
            if (p.test_stall && !wait_bar_warp(drain_bar(mw), 0u, abort_flag, p.err, false)) aborted = true;
            for (int u = u0; u < p.total_units && !aborted; u += ustep, ++tile_i) {
                const int acc = tile_i & 1;
                const uint32_t aph = (tile_i >> 1) & 1u;
                int next_key = key + kstep;
                if (next_key >= KT) next_key -= KT;
                if (u + ustep >= p.total_units) next_key = -1;
                if (!wait_bar_warp(tempty_bar(acc), aph ^ 1u, abort_flag, p.err, msleep)) {
                    aborted = true;
                    break;
                }
                if (resident && key != prev) {
                    if (!wait_bar_warp(full_b(0), jw & 1u, abort_flag, p.err, msleep)) {
                        aborted = true;
                        break;
                    }
                    ++jw;
                    prev = key;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NACC * BN) + (uint32_t)(mw * BN);
                uint32_t first = 1;
                for (int kg = 0; kg < p.slab_nkg && !aborted; ++kg, ra.next()) {
                    const int sa = ra.s;
                    if (!wait_bar_warp(full_a(sa), ra.ph, abort_flag, p.err, msleep)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a0 = sA + sa * a_stage + (uint32_t)(mw * p.slab_pair_rows) * 128u;
                    for (int bg = 0; bg < nbg; ++bg) {
                        uint32_t b0;
                        int sb = 0;
                        if (resident) {
                            b0 = sB + (uint32_t)(kg * nbg + bg) * b_stage;
                        } else {
                            sb = rb.s;
                            const uint32_t phb = rb.ph;
                            rb.next();
                            if (!wait_bar_warp(full_b(sb), phb, abort_flag, p.err, msleep)) {
                                aborted = true;
                                break;
                            }
                            tc_fence_after();
                            b0 = sB + sb * b_stage;
                        }
                        for (int t = 0; t < btaps; ++t) {
                            const uint32_t row = (uint32_t)(bg * g.dh * p.slab_bws + t * g.dw);
                            const uint64_t bd = sw128_desc(b0 + t * B_HALF);
                            const uint64_t ad = sw128_desc(a0 + row * 128u);
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                sp_mma_warp(d_tmem, ad + 2u * k, bd + 2u * k, IDESC, (first && k == 0) ? 0u : 1u);
                            first = 0;
                        }
                        if (!resident) sp_commit_warp(empty_b(sb));
                    }
                    sp_commit_warp(empty_a(sa));
                }
                if (aborted) break;
                if (resident && next_key != key) sp_commit_warp(empty_b(0));
                sp_commit_warp(tfull_bar(acc));
                key = next_key;
            }
            if (aborted) {
                sp_commit_local_warp(drain_bar(mw));
                if (lane == 0) {
                    const unsigned long long t0 = globaltimer();
                    while (!mbar_try_wait(drain_bar(mw), 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {}
                }
            } else {
                // every epilogue arrival (the peer's are remote) has landed before the leader leaves
                for (uint32_t t = tile_i; t < tile_i + 2u; ++t)
                    if (!wait_bar_warp(tempty_bar(t & 1), ((t >> 1) & 1u) ^ 1u, abort_flag, p.err, false)) break;
            }
        }
        __syncwarp();
    } else if (warp < EPI_WARPS) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int wq = warp & 3;
        constexpr int SCOLS = BN / 2 < 16 ? 16 : BN / 2;
        const int cb_begin = (warp >> 2) * SCOLS;
        const int cb_end = cb_begin + SCOLS < BN ? cb_begin + SCOLS : BN;
        const bool add_bias = p.epi == EPI_BIAS || p.epi == EPI_BIAS_GELU;
        const bool do_gelu = p.epi == EPI_BIAS_GELU || p.epi == EPI_GELU;
        uint8_t* stg = smem + stg_off + warp * STG_W;
        const uint32_t tempty_leader0 = cluster_map(tempty_bar(0), 0u);
        if (p.pdl) griddep_wait();
        uint32_t tile_i = 0;
        for (int u = u0; u < p.total_units; u += ustep, ++tile_i) {
            int mt, gi, nt;
            unit_tile(u, mt, gi, nt);
            const int acc = tile_i & 1;
            const uint32_t aph = (tile_i >> 1) & 1u;
            const TileOrigin to = tile_origin(p, mt);
            long long roff[NACC][EPI_MAX_LPR];
#pragma unroll
            for (int j = 0; j < NACC; ++j) {
                auto row_offset = [&](int rr) -> long long {
                    const int rh = fdiv(rr, p.f_bws), rw = rr - rh * p.slab_bws;
                    const int oh = to.oh0 + j * p.acc_bh + rh, ow = to.ow0 + rw;
                    if (rh >= p.acc_bh || rw >= p.BW || oh >= g.Ho || ow >= g.Wo || to.n >= g.N) return -1;
                    return (long long)(((to.n * g.Do + to.od) * g.Ho + oh) * g.Wo + ow) * (g.G * g.K);
                };
                epilogue_rows<SCOLS, 2>(lane, wq, row_offset, roff[j]);
            }
            if (!wait_bar_warp(tfull_bar(acc), aph, abort_flag, p.err, (p.sleep_mask & 2) != 0)) break;
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < NACC; ++j) {
                const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)((acc * NACC + j) * BN);
                epilogue_chunks<BN, SCOLS, 2>(p, taddr, lane, wq, cb_begin, cb_end, nt, gi, 0, false, add_bias, do_gelu,
                                              stg, roff[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(tempty_bar(acc));
                else sp_arrive_cluster(tempty_leader0 + 8u * (uint32_t)acc);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();
    if (warp == SP_MMA_WARP) {
        tc_fence_after();
        sp_tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int BN, int BY, int BT, int NACC>
cudaError_t launch_slab_pair_one(const TcParams& p, const CUtensorMap& amap, const CUtensorMap& wmap, int grid,
                                 size_t smem, cudaStream_t stream) {
    auto kern = conv_fwd_slab_pair_kernel<BN, BY, BT, NACC>;
    static bool attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SLAB_SMEM_MAX);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    return launch_kernel(kern, dim3(grid), dim3(SP_THREADS), smem, stream, p.pdl != 0, 2, p, amap, wmap);
}

}  // namespace

size_t slab_pair_smem_bytes(int BN, int sa, int sb, size_t a_stage, int btaps) {
    const size_t b_stage = (size_t)btaps * (BN / 2) * 128;
    return 1024 + (size_t)sa * a_stage + (size_t)sb * b_stage + (size_t)EPI_WARPS * slab_stg_warp_bytes(BN, 2) +
           8 * (2 * SP_MAX_SA + 2 * SP_MAX_SB + 6) + 16;
}

int slab_pair_max_clusters(size_t smem) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(SP_THREADS);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    auto kern = conv_fwd_slab_pair_kernel<64, 3, 3, 2>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SLAB_SMEM_MAX) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

cudaError_t launch_slab_pair(const TcParams& p, const CUtensorMap* act_map, const CUtensorMap* w_map, int grid,
                             size_t smem, cudaStream_t stream) {
    if (!act_map || !w_map || p.tf32 || p.lat.on || p.slab_nacc < 1 || p.slab_nacc > 2 || (grid & 1) || p.slab_sa < 2 ||
        p.slab_sa > SP_MAX_SA || (!p.slab_resident && (p.slab_sb < 2 || p.slab_sb > SP_MAX_SB)) ||
        smem > SLAB_SMEM_MAX)
        return cudaErrorInvalidValue;
#define X(bn, nacc)                                                                                     \
    if (p.BN == bn && p.slab_nacc == nacc) {                                                            \
        if (p.slab_btaps == 3 && p.slab_nbg == 3)                                                       \
            return launch_slab_pair_one<bn, 3, 3, nacc>(p, *act_map, *w_map, grid, smem, stream);       \
        return launch_slab_pair_one<bn, 0, 0, nacc>(p, *act_map, *w_map, grid, smem, stream);           \
    }
    X(32, 2) X(64, 2) X(32, 1) X(64, 1)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace convfwd
