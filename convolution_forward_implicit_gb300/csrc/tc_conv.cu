// Implicit-GEMM convolution forward on the sm_103a tensor cores (tcgen05), fp32
// accumulation in tensor memory, fused bias + GELU epilogue.  bf16 I/O multiplies bf16
// operands (kind::f16); fp32 I/O runs as 3xTF32 (kind::tf32): every fp32 operand is split
// into an exactly-TF32 high part and a low remainder, and three TF32 products (lo*hi,
// hi*lo, hi*hi) recover fp32-level products.
//
// GEMM view per group g (page "composable_kernel ... LEARNINGS_GROUPED_CONV.md",
// introduction: NHWGC x GKYXC -> NHWGK): rows m are output pixels (n, od, oh, ow),
// columns are output channels k, and the reduction runs over (tap, c) with c innermost,
// so that one 16-byte chunk of the reduction is 8 consecutive channels of one input
// pixel.  The im2col matrix of page "[ET-VK] conv1d runs at ~3% ...", section "The
// conv2d path already solves this", is never materialised: each A tile is gathered
// straight from the channels-last input, zero-filled where a tap falls in the padding.
//
// One persistent CTA per SM (grid = min(units, SMs)), warp-specialised (EW = 8 or 16
// epilogue warps):
//   warps 0..EW-1   epilogue: EW/4 warps per TMEM lane quarter (warp w owns lanes
//               32(w%4)..+31 and a 1/(EW/4) share of the columns); tcgen05.ld, bias, GELU,
//               rounding, then stores through a per-warp staging buffer so each store
//               instruction writes whole row segments (fp32 partial sums instead when the
//               reduction is split).
//   next 4 warps (3 with EW = 16)   producers, per K block (one tap x 64 bf16 or 32 fp32
//               channels): TMA gather: one 5-D tiled box of BH x BW output pixels (conv stride
//               as the element stride, padding as out-of-bounds zero fill) plus one bulk copy
//               of the prepacked weight tile, issued by the warp that owns the stage;
//               cp.async gather: 16-byte zero-filling copies of 8-channel chunks packed
//               densely across taps, for channel counts no box can serve.
//   next warp   MMA: one thread issues tcgen05.mma (M = 128, N = BN; 4 x K=16 bf16 or
//               12 x K=8 tf32 per K block) and tcgen05.commit frees the stage; the
//               accumulator is double-buffered in TMEM so the epilogue of tile i overlaps
//               the main loop of tile i+1.
//   last 4 warps (3xTF32 only) split each activation tile into hi and lo parts in place.
// Every mbarrier wait is bounded: after ~1 s it raises the device error word, sets a
// CTA-wide abort flag and the CTA winds down (drains copies, waits for issued MMAs,
// frees TMEM).
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "tc_common.cuh"

namespace convfwd {
namespace {
// Kernel kinds: bf16 operands gathered by cp.async (any C multiple of 8), bf16 gathered by
// TMA boxes, and fp32 I/O as three TF32 products per useful product (3xTF32, TMA gather).
enum Kind { KIND_BF16_CPASYNC = 0, KIND_BF16_TMA = 1, KIND_TF32X3 = 2 };

// A thread has at most one TMA copy in flight (measured on this GPU: a second copy from the
// same thread starts only when the first completes, ~700 cycles each), so the TMA producer
// spreads its copies over 4 warps, pipeline stage s belonging to warp s % 4, where lane 0
// copies the activation box and lane 1 the weight tile.  With 16 epilogue warps there are 3
// producer warps (those plans have 3 or 5 stages): 20 warps in all leave each SM sub-partition
// 5 warps, so a thread may hold 96 registers (21 warps: 6 on one sub-partition, 80 registers).
template <int KIND, int EW>
struct Traits {
    static constexpr bool TMA = KIND != KIND_BF16_CPASYNC;
    static constexpr bool TF32 = KIND == KIND_TF32X3;
    static constexpr int PROD_WARPS = EW == 16 ? 3 : 4;
    static constexpr int CVT_WARPS = TF32 ? 4 : 0;
    static constexpr int MMA_WARP = EW + PROD_WARPS;
    static constexpr int CVT_WARP0 = MMA_WARP + 1;
    static constexpr int THREADS = (CVT_WARP0 + CVT_WARPS) * 32;
    static constexpr int PROD_THREADS = PROD_WARPS * 32;
    static constexpr uint32_t FULL_COUNT = TMA ? 1u : (uint32_t)(PROD_THREADS + 1);
    static constexpr uint32_t A_STAGE = TF32 ? 2 * A_BYTES : A_BYTES;   // 3xTF32: hi tile, then lo tile
};

template <int BN, int KIND>
struct Cfg {
    static constexpr uint32_t B_TILE = BN * 128;
    static constexpr uint32_t B_STAGE = KIND == KIND_TF32X3 ? 2 * B_TILE : B_TILE;
    static constexpr uint32_t TMEM_COLS = (2 * BN < 32) ? 32 : 2 * BN;    // power of two for BN in {16..256}
};

// Shared memory of one configuration: 1 KB alignment slack, the ring, the epilogue staging,
// then (16 epilogue warps with bf16 outputs, where it fits) each epilogue warp's bias columns
// in fp32, then the barriers.  With 16 warps every lane of a warp needs the same bias values,
// so the warp converts its columns once per tile instead of each lane once per output.
template <int BN, int STAGES, int KIND, int EW>
struct Smem {
    static constexpr size_t LIMIT = 232448;
    static constexpr size_t RING = (size_t)STAGES * (Traits<KIND, EW>::A_STAGE + Cfg<BN, KIND>::B_STAGE);
    static constexpr size_t STG_W = STG_WARP_BYTES;   // staging per epilogue warp
    static constexpr size_t STG = (size_t)EW * STG_W;
    static constexpr size_t BARS = 8 * (3 * STAGES + 5) + 16;
    static constexpr size_t BIAS_NEED = (size_t)16 * BN;   // EW warps x BN/(EW/4) columns x 4 bytes
    static constexpr bool BIAS_SMEM =
        EW == 16 && KIND == KIND_BF16_TMA && 1024 + RING + STG + BIAS_NEED + BARS <= LIMIT;
    static constexpr size_t BIAS_BYTES = BIAS_SMEM ? BIAS_NEED : 0;
    static constexpr size_t TOTAL = 1024 + RING + STG + BIAS_BYTES + BARS;
};

// MC: the CTAs run as clusters of two that compute the tiles 2j and 2j+1 along M of the same
// (group, N tile) in lockstep; each loads one half of every weight tile and multicasts it to
// both, so the pair reads each weight tile from L2 once instead of twice.  A stage is then
// refilled only after the MMAs of both CTAs have released it (each CTA's commits arrive on
// the empty barriers of both).
template <int BN, int STAGES, int KIND, int EW, bool MC>
__global__ void __launch_bounds__(Traits<KIND, EW>::THREADS, 1)
    conv_fwd_tc_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap act_map,
                       const __grid_constant__ CUtensorMap y_map) {
    using C = Cfg<BN, KIND>;
    using T = Traits<KIND, EW>;
    static_assert(!MC || KIND == KIND_BF16_TMA, "weight multicast is built for the bf16 TMA kernel");
    constexpr int RED_PITCH = BN + 4;   // floats per row of the cluster-reduction buffer
    static_assert((size_t)BM * RED_PITCH * 4 <= (size_t)STAGES * (T::A_STAGE + C::B_STAGE),
                  "the cluster-reduction buffer reuses the stage area");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const uint32_t sA = sbase;
    const uint32_t sB = sbase + STAGES * T::A_STAGE;
    using SM = Smem<BN, STAGES, KIND, EW>;
    constexpr uint32_t STG_OFFSET = STAGES * (T::A_STAGE + C::B_STAGE);       // epilogue staging
    constexpr uint32_t BIAS_OFFSET = STG_OFFSET + (uint32_t)SM::STG;          // fp32 bias columns
    const uint32_t bar0 = sbase + BIAS_OFFSET + (uint32_t)SM::BIAS_BYTES;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    auto cvt_bar = [&](int s) { return bar0 + 8u * (2 * STAGES + s); };
    auto tfull_bar = [&](int a) { return bar0 + 8u * (3 * STAGES + a); };
    auto tempty_bar = [&](int a) { return bar0 + 8u * (3 * STAGES + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (3 * STAGES + 4);
    uint8_t* misc = smem + (bar0 + 8u * (3 * STAGES + 5) - sbase);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), T::FULL_COUNT);
            mbar_init(empty_bar(s), MC ? 2 : 1);
            mbar_init(cvt_bar(s), T::CVT_WARPS > 0 ? T::CVT_WARPS : 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), 1);
            mbar_init(tempty_bar(a), EW);
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (T::TMA && warp == EW && lane == 0)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&act_map)) : "memory");
    if (warp == T::MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // the peer CTA's copies and commits reach this CTA's barriers only after both are set up
    if (MC) cluster_sync_all();
    // set up: the next kernel on the stream may start (its own set-up and weight loads)
    if (p.pdl) griddep_launch();

    const Geom& g = p.g;
    const int GC = g.G * g.C;
    const int GK = g.G * g.K;
    // units of this CTA: u0, u0 + ustep, ...; with MC a unit is a pair of M tiles (the CTA of
    // cluster rank r takes tile 2 mt + r of it)
    const uint32_t crank = MC ? cluster_ctarank() : 0u;
    const int u0 = MC ? (int)(blockIdx.x >> 1) : (int)blockIdx.x;
    const int ustep = MC ? (int)(gridDim.x >> 1) : (int)gridDim.x;
    auto unit_tile = [&](int u, int& mt, int& gi, int& nt, int& split) {
        decode_unit(p, u, mt, gi, nt, split);
        if (MC) mt = 2 * mt + (int)crank;
    };

    if (warp >= EW && warp < T::MMA_WARP) {
        const uint8_t* wp = reinterpret_cast<const uint8_t*>(p.wpack);
        if (T::TMA) {
            // -------------------------------------------------------- producer (TMA)
            const int pw = warp - EW;
            if (lane < 2) {
                const uint32_t a_tx = (uint32_t)(p.BW * p.BH) * 128u;
                const int cblk = T::TF32 ? 32 : 64;     // channels in one 128-byte row
                uint32_t it = 0, issued = 0;   // issued: 1 + the last iteration this warp loaded
                bool aborted = false;
                bool x_ready = !p.pdl;      // x may come from the previous kernel on the stream
                if (!x_ready && lane == 0 && u0 < p.total_units) {
                    // this warp's activation boxes of the first unit's first stages go into L2
                    // while the previous kernel finishes
                    int mt, gi, nt, split;
                    unit_tile(u0, mt, gi, nt, split);
                    if (mt < p.num_mt) {
                        const TileOrigin to = tile_origin(p, mt);
                        const int kb0 = split * p.kbps, kb1 = min(kb0 + p.kbps, p.nkb);
                        for (int kb = kb0 + pw; kb < kb1 && kb < kb0 + STAGES; kb += T::PROD_WARPS) {
                            const int tap = fdiv(kb, p.f_cbt);
                            const int c0 = (kb - tap * p.cbt) * cblk;
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
                    // (with MC the second tile of the last pair may lie past the output: its boxes
                    // are then out of range and read zeros, and the epilogue stores nothing)
                    const TileOrigin to = tile_origin(p, mt);
                    const int kb0 = split * p.kbps;
                    const int kb1 = min(kb0 + p.kbps, p.nkb);
                    const int w0 = to.ow0 * g.sw - g.pw, h0 = to.oh0 * g.sh - g.ph, d0 = to.od * g.sd - g.pd;
                    for (int kb = kb0; kb < kb1; ++kb, ++it) {
                        // stage s belongs to producer warp s % PROD_WARPS: a warp then refills a
                        // stage only after it has seen the stage's previous phase complete, so no
                        // parity wait is ever more than one phase ahead of its barrier
                        if ((int)((it % STAGES) % T::PROD_WARPS) != pw) continue;
                        const int s = it % STAGES;
                        const uint32_t ph = (it / STAGES) & 1u;
                        // lane 0 waits and both lanes follow its outcome, so they never part ways
                        int ok = 1;
                        if (lane == 0) ok = wait_bar(empty_bar(s), ph ^ 1u, abort_flag, p.err, p.sleep_mask & 1) ? 1 : 0;
                        ok = __shfl_sync(0x3u, ok, 0);
                        if (!ok) { aborted = true; break; }
                        if (lane == 0) mbar_arrive_expect_tx(full_bar(s), a_tx + C::B_STAGE);
                        issued = it + 1;
                        __syncwarp(0x3u);
                        if (lane == 0) {
                            if (!x_ready) {
                                griddep_wait();
                                x_ready = true;
                            }
                            const int tap = fdiv(kb, p.f_cbt);
                            const int c0 = (kb - tap * p.cbt) * cblk;
                            const int zz = fdiv(tap, p.f_YX);
                            const int rem = tap - zz * g.Y * g.X;
                            const int yy = fdiv(rem, p.f_X);
                            const int xx = rem - yy * g.X;
                            const int wi = w0 + xx * g.dw, hi = h0 + yy * g.dh;
                            if (p.map_kind == 0)
                                tma_load_5d(sA + s * T::A_STAGE, &act_map, gi * g.C + c0, wi, hi, d0 + zz * g.dd,
                                            to.n, full_bar(s));
                            else
                                tma_load_5d(sA + s * T::A_STAGE, &act_map, c0, gi, wi, hi, to.n, full_bar(s));
                        } else {
                            const size_t off = ((size_t)(gi * p.num_nt + nt) * p.nkb + kb) * C::B_STAGE;
                            if (MC) {
                                // this CTA's half of the weight tile (BN/2 rows), to both CTAs
                                constexpr uint32_t HALF = C::B_STAGE / 2;
                                bulk_g2s_multicast(sB + s * C::B_STAGE + crank * HALF, wp + off + crank * HALF, HALF,
                                                   full_bar(s), (uint16_t)0x3);
                            } else {
                                bulk_g2s(sB + s * C::B_STAGE, wp + off, C::B_STAGE, full_bar(s));
                            }
                        }
                    }
                }
                if (MC && lane == 0) {
                    // before the CTA may exit, every commit the peer's MMA role sends to this CTA's
                    // empty barriers must have arrived: wait (bounded) for the phases that would
                    // precede this warp's next STAGES refills
                    for (uint32_t k = it; k < it + (uint32_t)STAGES; ++k)
                        if ((int)((k % STAGES) % T::PROD_WARPS) == pw &&
                            !wait_bar(empty_bar(k % STAGES), ((k / STAGES) & 1u) ^ 1u, abort_flag, p.err, false))
                            break;
                }
                if (aborted && lane == 0) {
                    // before the CTA exits, the copies this warp issued into stages the MMA role never
                    // consumed must have landed: a bounded wait on each of its last ring pass's stages
                    const unsigned long long t0 = globaltimer();
                    for (uint32_t k = issued > (uint32_t)STAGES ? issued - STAGES : 0u; k < issued; ++k)
                        if ((int)((k % STAGES) % T::PROD_WARPS) == pw)
                            while (!mbar_try_wait(full_bar(k % STAGES), (k / STAGES) & 1u) &&
                                   globaltimer() - t0 < WAIT_LIMIT_NS) {
                            }
                }
            }
            __syncwarp();
        } else {
            // -------------------------------------------------------- producer (cp.async)
            const int pt = threadIdx.x - EW * 32;
            const int j = pt & 7;        // 16-byte chunk of the 128-byte row
            const int rb = pt >> 3;      // rows rb, rb+16, ..., rb+112
            const uint32_t swz = (uint32_t)((j ^ (rb & 7)) << 4);
            const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(p.x);
            if (p.pdl) griddep_wait();
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
                        const int t1 = fdiv(m, p.f_Wo);
                        const int ow = m - t1 * g.Wo;
                        const int t2 = fdiv(t1, p.f_Ho);
                        const int oh = t1 - t2 * g.Ho;
                        rn[i] = fdiv(t2, p.f_Do);
                        const int od = t2 - rn[i] * g.Do;
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
                    if (!wait_bar(empty_bar(s), ph ^ 1u, abort_flag, p.err, p.sleep_mask & 1)) { aborted = true; break; }
                    if (pt == 0) {
                        mbar_arrive_expect_tx(full_bar(s), C::B_STAGE);
                        const size_t off = ((size_t)(gi * p.num_nt + nt) * p.nkb + kb) * C::B_STAGE;
                        bulk_g2s(sB + s * C::B_STAGE, wp + off, C::B_STAGE, full_bar(s));
                    }
                    const int q = kb * 8 + j;
                    const bool qok = q < p.nchunks;
                    const int tap = qok ? fdiv(q, p.f_cpt) : 0;
                    const int c0 = (q - tap * p.cpt) * 8;
                    const int zz = fdiv(tap, p.f_YX);
                    const int rem = tap - zz * g.Y * g.X;
                    const int yy = fdiv(rem, p.f_X);
                    const int xx = rem - yy * g.X;
                    const int dz = zz * g.dd, dy = yy * g.dh, dx = xx * g.dw;
                    const uint32_t dst0 = sA + s * T::A_STAGE + swz;
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
        }
    } else if (warp == T::MMA_WARP) {
        // ------------------------------------------------------------ MMA issue
        // bounded waits start once the previous kernel on the stream has completed
        if (p.pdl) griddep_wait();
        if (lane == 0) {
            constexpr uint32_t IDESC = idesc_f32acc(BM, BN, T::TF32 ? 2u : 1u);
            uint32_t it = 0, tile_i = 0;
            bool aborted = false;
            // test hook: wait on a barrier nothing completes, so the bounded wait runs out and
            // the abort path (error word, drained copies, freed tensor memory) is exercised
            if (p.test_stall && !wait_bar(drain_bar, 0u, abort_flag, p.err, false)) aborted = true;
            for (int u = u0; u < p.total_units && !aborted; u += ustep, ++tile_i) {
                int mt, gi, nt, split;
                unit_tile(u, mt, gi, nt, split);
                const int kb0 = split * p.kbps;
                const int kb1 = min(kb0 + p.kbps, p.nkb);
                const int acc = tile_i & 1;
                const uint32_t aph = (tile_i >> 1) & 1u;
                if (!wait_bar(tempty_bar(acc), aph ^ 1u, abort_flag, p.err, (p.sleep_mask & 4) != 0)) { aborted = true; break; }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t ph = (it / STAGES) & 1u;
                    if (!wait_bar(T::TF32 ? cvt_bar(s) : full_bar(s), ph, abort_flag, p.err, (p.sleep_mask & 4) != 0)) {
                        aborted = true;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t ad = sw128_desc(sA + s * T::A_STAGE);
                    const uint64_t bd = sw128_desc(sB + s * C::B_STAGE);
                    if (T::TF32) {
                        // hi tiles first in the stage, lo tiles after: +A_BYTES / +B_TILE bytes
                        const uint64_t alo = ad + (A_BYTES >> 4), blo = bd + (C::B_TILE >> 4);
#pragma unroll
                        for (int k = 0; k < 4; ++k) {   // 4 x K=8 tf32 = 32 fp32 = one 128-byte row
                            mma_tf32(d_tmem, alo + 2u * k, bd + 2u * k, IDESC, (kb > kb0 || k > 0) ? 1u : 0u);
                            mma_tf32(d_tmem, ad + 2u * k, blo + 2u * k, IDESC, 1u);
                            mma_tf32(d_tmem, ad + 2u * k, bd + 2u * k, IDESC, 1u);
                        }
                    } else {
                        mma_bf16_k4(d_tmem, ad, bd, IDESC, kb > kb0 ? 1u : 0u);   // 4 x K=16 = one 128-byte row
                    }
                    if (MC) mma_commit_multicast(empty_bar(s), (uint16_t)0x3);   // both CTAs' copy of the stage
                    else mma_commit(empty_bar(s));
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
    } else if (T::TF32 && warp >= T::CVT_WARP0) {
        // ------------------------------------------------------------ hi/lo split (3xTF32)
        if (p.pdl) griddep_wait();
        // Every fp32 activation x splits into hi = x with its low 13 mantissa bits cleared (exact
        // in TF32) and lo = x - hi (exact in fp32); the MMA then sums lo*w_hi + hi*w_lo + hi*w_hi.
        // hi is the tile as the TMA wrote it: kind::tf32 reads an fp32 operand by ignoring those
        // 13 bits (measured: every product equals the truncated operand's), so only lo is written.
        const int ct = threadIdx.x - T::CVT_WARP0 * 32;
        const int n16 = p.BW * p.BH * 8;   // 16-byte chunks the TMA box wrote
        uint32_t it = 0;
        bool aborted = false;
        for (int u = blockIdx.x; u < p.total_units && !aborted; u += gridDim.x) {
            int mt, gi, nt, split;
            decode_unit(p, u, mt, gi, nt, split);
            const int kb0 = split * p.kbps;
            const int kb1 = min(kb0 + p.kbps, p.nkb);
            for (int kb = kb0; kb < kb1; ++kb, ++it) {
                const int s = it % STAGES;
                const uint32_t ph = (it / STAGES) & 1u;
                if (!wait_bar_warp(full_bar(s), ph, abort_flag, p.err, (p.sleep_mask & 8) != 0)) { aborted = true; break; }
                uint4* hi = reinterpret_cast<uint4*>(smem + s * T::A_STAGE);
                uint4* lo = reinterpret_cast<uint4*>(smem + s * T::A_STAGE + A_BYTES);
                for (int i = ct; i < n16; i += T::CVT_WARPS * 32) {
                    const uint4 v = hi[i];
                    uint4 h, l;
                    h.x = v.x & 0xFFFFE000u; h.y = v.y & 0xFFFFE000u; h.z = v.z & 0xFFFFE000u; h.w = v.w & 0xFFFFE000u;
                    l.x = __float_as_uint(__uint_as_float(v.x) - __uint_as_float(h.x));
                    l.y = __float_as_uint(__uint_as_float(v.y) - __uint_as_float(h.y));
                    l.z = __float_as_uint(__uint_as_float(v.z) - __uint_as_float(h.z));
                    l.w = __float_as_uint(__uint_as_float(v.w) - __uint_as_float(h.w));
                    lo[i] = l;
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(cvt_bar(s));
            }
        }
    } else if (warp < EW) {
        // ------------------------------------------------------------ epilogue
        // Warp w owns the 32 accumulator rows of TMEM lane quarter w % 4 and half of the
        // columns.  It works in chunks of columns that make one output row segment of at most
        // 128 bytes: read TMEM, add bias, GELU, convert, and write its 32 row segments into a
        // shared staging buffer (16-byte slots XOR-swizzled by row: conflict-free both ways);
        // then the warp reads the buffer back row-wise and stores whole row segments, so one
        // store instruction writes 4 full 128-byte segments instead of 32 scattered 16-byte
        // pieces.  Split plans store fp32 partial sums to the workspace the same way.
        const int wq = warp & 3;
        constexpr int COLS = BN / (EW / 4) < 16 ? 16 : BN / (EW / 4);   // EW/4 warps share a lane quarter
        constexpr int CC2 = COLS, CC4 = COLS;   // columns per staged chunk: bf16, fp32 outputs
        const int cb_begin = (warp >> 2) * COLS;
        const int cb_end = cb_begin + COLS < BN ? cb_begin + COLS : BN;
        const bool partial = p.splits > 1;
        const bool add_bias = (p.epi == EPI_BIAS || p.epi == EPI_BIAS_GELU) && !partial;
        const bool do_gelu = (p.epi == EPI_BIAS_GELU || p.epi == EPI_GELU) && !partial;
        uint8_t* stg = smem + STG_OFFSET + warp * (uint32_t)SM::STG_W;
        if (p.pdl) griddep_wait();   // y, the workspace and bias may belong to the previous kernel
        uint32_t tile_i = 0;
        for (int u = u0; u < p.total_units; u += ustep, ++tile_i) {
            int mt, gi, nt, split;
            unit_tile(u, mt, gi, nt, split);
            const int acc = tile_i & 1;
            const uint32_t aph = (tile_i >> 1) & 1u;
            TileOrigin to{0, 0, 0, 0};
            if (T::TMA) to = tile_origin(p, mt);
            // element offset of accumulator row rr's pixel, or -1 if the row is outside the output
            // (p.lat is the identity placement unless final outputs land on a lattice of y; the
            // host passes the identity to kernels that write partial sums)
            auto row_offset = [&](int rr) -> long long {
                if (T::TMA) {
                    const int rh = fdiv(rr, p.f_BW);
                    const int oh = to.oh0 + rh, ow = to.ow0 + (rr - rh * p.BW);
                    if (rr >= p.BW * p.BH || oh >= g.Ho || ow >= g.Wo || (MC && to.n >= g.N)) return -1;
                    return (long long)lattice_pixel(p.lat, to.n, to.od, oh, ow) * GK;
                }
                const int m = mt * BM + rr;
                if (m >= g.M) return -1;
                return (p.lat.on ? out_pixel_linear(p, m) : (long long)m) * GK;
            };
            if (p.cluster_red) {
                // one unit per CTA: its partial accumulator goes to this CTA's shared memory
                // (the drained stage area, row pitch BN + 4 floats), for the cluster reduction
                // after the role loops
                if (!wait_bar_warp(tfull_bar(acc), aph, abort_flag, p.err, (p.sleep_mask & 2) != 0)) break;
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * BN);
                float* red_row = reinterpret_cast<float*>(smem) + (size_t)(wq * 32 + lane) * RED_PITCH;
                for (int cb = cb_begin; cb < cb_end; cb += 16) {
                    uint32_t v[16];
                    __syncwarp();
                    tmem_ld16(taddr + (uint32_t)cb, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<uint4*>(red_row + cb + e) = make_uint4(v[e], v[e + 1], v[e + 2], v[e + 3]);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(tempty_bar(acc));
                continue;
            }
            const bool wide = partial || T::TF32;     // fp32 stores
            long long roff[EPI_MAX_LPR];
            if (wide) epilogue_rows<CC4, 4>(lane, wq, row_offset, roff);
            else epilogue_rows<CC2, 2>(lane, wq, row_offset, roff);
            float* bsm = nullptr;
            if (SM::BIAS_SMEM && add_bias) {
                // this warp's bias columns of tile nt in fp32 (columns past K as zeros, never
                // stored); the warp's previous tile has finished reading them
                bsm = reinterpret_cast<float*>(smem + BIAS_OFFSET) + warp * COLS;
                const __nv_bfloat16* bias = reinterpret_cast<const __nv_bfloat16*>(p.bias) + (size_t)gi * g.K;
                for (int c = 2 * lane; c < cb_end - cb_begin; c += 64) {
                    const int n = nt * BN + cb_begin + c;
                    float2 bf = make_float2(0.f, 0.f);
                    if (n < g.K) {
                        const uint32_t w2 = __ldg(reinterpret_cast<const unsigned int*>(bias + n));
                        bf = make_float2(__uint_as_float(w2 << 16), __uint_as_float(w2 & 0xFFFF0000u));
                    }
                    *reinterpret_cast<float2*>(bsm + c) = bf;
                }
                __syncwarp();
            }
            if (!wait_bar_warp(tfull_bar(acc), aph, abort_flag, p.err, (p.sleep_mask & 2) != 0)) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)(acc * BN);
            if (wide)
                epilogue_chunks<BN, CC4, 4, EW == 8>(p, taddr, lane, wq, cb_begin, cb_end, nt, gi, split, partial, add_bias,
                                       do_gelu, stg, roff);
            else
                epilogue_chunks<BN, CC2, 2, EW == 8>(p, taddr, lane, wq, cb_begin, cb_end, nt, gi, split, partial, add_bias,
                                       do_gelu, stg, roff, bsm, (T::TMA && p.ystore) ? &y_map : nullptr,
                                       YBox{to.ow0 + wq * 32, to.oh0, to.od, to.n});
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
        }
        // the tensor-map stores have completed before this CTA may leave
        if (p.ystore && lane == 0) bulk_wait_all();
        __syncwarp();
    }

    if (p.cluster_red) {
        // Split-K reduction across the cluster (the p.splits CTAs of one tile, cluster rank =
        // split): once every partial sits in its CTA's shared memory, CTA k sums rows
        // [k R, (k+1) R) of all partials in split order (so the result does not depend on
        // timing), adds bias, applies GELU and stores y.  A second cluster barrier keeps each
        // CTA's buffer alive until the others have read it.
        cluster_sync_all();
        if (warp < EW && blockIdx.x < (unsigned)p.total_units) {
            int mt, gi, nt, split;
            decode_unit(p, blockIdx.x, mt, gi, nt, split);
            TileOrigin to{0, 0, 0, 0};
            if (T::TMA) to = tile_origin(p, mt);
            const int S = p.splits;
            const int R = BM / S;
            const int r0 = (int)cluster_ctarank() * R;
            const bool add_bias = p.epi == EPI_BIAS || p.epi == EPI_BIAS_GELU;
            const bool do_gelu = p.epi == EPI_BIAS_GELU || p.epi == EPI_GELU;
            const uint32_t red0 = smem_u32(smem);
            const int per_row = BN / 4;
            for (int i = threadIdx.x; i < R * per_row; i += EW * 32) {
                const int rr = r0 + i / per_row;
                const int col = (i - (i / per_row) * per_row) * 4;
                const int n = nt * BN + col;
                if (n >= g.K) continue;
                long long m;
                if (T::TMA) {
                    const int rh = fdiv(rr, p.f_BW);
                    const int oh = to.oh0 + rh, ow = to.ow0 + (rr - rh * p.BW);
                    if (rr >= p.BW * p.BH || oh >= g.Ho || ow >= g.Wo) continue;
                    m = lattice_pixel(p.lat, to.n, to.od, oh, ow);
                } else {
                    const int ml = mt * BM + rr;
                    if (ml >= g.M) continue;
                    m = p.lat.on ? out_pixel_linear(p, ml) : ml;
                }
                const uint32_t off = (uint32_t)(rr * RED_PITCH + col) * 4u;
                // all S partials requested before the first add, so their latencies overlap
                float4 pv[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    if (j < S) pv[j] = ld_cluster_f4(cluster_map(red0 + off, (uint32_t)j));
                float4 a = pv[0];
#pragma unroll
                for (int j = 1; j < 8; ++j)
                    if (j < S) { a.x += pv[j].x; a.y += pv[j].y; a.z += pv[j].z; a.w += pv[j].w; }
                float v[4] = {a.x, a.y, a.z, a.w};
                const size_t o = (size_t)m * GK + (size_t)gi * g.K + n;
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (add_bias) {
                        v[e] += T::TF32 ? reinterpret_cast<const float*>(p.bias)[(size_t)gi * g.K + n + e]
                                        : __bfloat162float(
                                              reinterpret_cast<const __nv_bfloat16*>(p.bias)[(size_t)gi * g.K + n + e]);
                    }
                    if (do_gelu) v[e] = gelu(v[e]);
                }
                if (T::TF32) {
                    *reinterpret_cast<float4*>(reinterpret_cast<float*>(p.y) + o) = make_float4(v[0], v[1], v[2], v[3]);
                } else {
                    *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(p.y) + o) =
                        make_uint2(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]));
                }
            }
        }
        cluster_sync_all();
    }

    tc_fence_before();
    __syncthreads();
    // no CTA of a pair leaves while the other may still copy into or arrive on its shared memory
    if (MC) cluster_sync_all();
    if (warp == T::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int BN, int STAGES, int KIND, int EW>
constexpr size_t smem_bytes_for() {
    return Smem<BN, STAGES, KIND, EW>::TOTAL;
}

template <int BN, int STAGES, int KIND, int EW, bool MC = false>
cudaError_t launch_one(const TcParams& p, const CUtensorMap& map, const CUtensorMap& ymap, int grid,
                       cudaStream_t stream) {
    auto kern = conv_fwd_tc_kernel<BN, STAGES, KIND, EW, MC>;
    constexpr size_t smem = smem_bytes_for<BN, STAGES, KIND, EW>();
    static_assert(smem <= 232448, "shared memory budget");
    // opt in to the large dynamic shared memory once per device (not inside graph capture)
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
    return launch_kernel(kern, dim3(grid), dim3(Traits<KIND, EW>::THREADS), smem, stream, p.pdl != 0,
                         MC ? 2 : p.cluster_red ? p.splits : 1, p, map, ymap);
}

}  // namespace

// (BN, stages) pairs compiled into the library, per kind and epilogue width; the plan picks one.
#define TC_BF16_CONFIGS(X) X(256, 4) X(128, 6) X(64, 8) X(32, 8) X(16, 8)
#define TC_BF16_EPI16_CONFIGS(X) X(256, 3) X(128, 5)
#define TC_TF32_CONFIGS(X) X(256, 2) X(128, 3) X(64, 4) X(32, 4) X(16, 5)
// weight multicast (bf16, 8 or 16 epilogue warps at the stage counts above)
#define TC_BF16_MC_CONFIGS(X) X(256, 4, 8) X(128, 6, 8) X(256, 3, 16) X(128, 5, 16)

int tc_stages_for(int BN, int tf32, int epi_warps) {
#define X(bn, st) if (BN == bn) return st;
    if (tf32) { TC_TF32_CONFIGS(X) }
    else if (epi_warps == 16) { TC_BF16_EPI16_CONFIGS(X) }
    else { TC_BF16_CONFIGS(X) }
#undef X
    return 0;
}

int tc_mc_max_clusters(int BN, int epi_warps) {
    const int st = tc_stages_for(BN, 0, epi_warps);
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
#define X(bn, stg, ew)                                                                                  \
    if (BN == bn && st == stg && epi_warps == ew)                                                       \
        return query(conv_fwd_tc_kernel<bn, stg, KIND_BF16_TMA, ew, true>, smem_bytes_for<bn, stg, KIND_BF16_TMA, ew>(), \
                     Traits<KIND_BF16_TMA, ew>::THREADS);
    TC_BF16_MC_CONFIGS(X)
#undef X
    return 0;
}

cudaError_t launch_tc(const TcParams& p, const CUtensorMap* act_map, const CUtensorMap* y_map, int stages, int grid,
                      cudaStream_t stream) {
    static const CUtensorMap unused{};
    const CUtensorMap& map = act_map ? *act_map : unused;
    const CUtensorMap& ymap = y_map ? *y_map : unused;
    if (p.tma && !act_map) return cudaErrorInvalidValue;
    if (p.ystore && (!y_map || !p.tma || p.tf32 || p.splits != 1 || p.lat.on || p.BH != 1 || p.BW % 32 != 0))
        return cudaErrorInvalidValue;
    if (p.tf32) {
        if (!p.tma || p.epi_warps != 8) return cudaErrorInvalidValue;
#define X(bn, st) \
    if (p.BN == bn && stages == st) return launch_one<bn, st, KIND_TF32X3, 8>(p, map, ymap, grid, stream);
        TC_TF32_CONFIGS(X)
#undef X
        return cudaErrorInvalidValue;
    }
    if (p.mc) {
        // pairs of CTAs: an even grid, one tile pair per unit, no split of the reduction
        if (!p.tma || p.splits != 1 || p.cluster_red || (grid & 1)) return cudaErrorInvalidValue;
#define X(bn, st, ew)                                                 \
    if (p.BN == bn && stages == st && p.epi_warps == ew)              \
        return launch_one<bn, st, KIND_BF16_TMA, ew, true>(p, map, ymap, grid, stream);
        TC_BF16_MC_CONFIGS(X)
#undef X
        return cudaErrorInvalidValue;
    }
    if (p.epi_warps == 16) {
        if (!p.tma) return cudaErrorInvalidValue;
#define X(bn, st) \
    if (p.BN == bn && stages == st) return launch_one<bn, st, KIND_BF16_TMA, 16>(p, map, ymap, grid, stream);
        TC_BF16_EPI16_CONFIGS(X)
#undef X
        return cudaErrorInvalidValue;
    }
    if (p.epi_warps != 8) return cudaErrorInvalidValue;
#define X(bn, st)                                                                              \
    if (p.BN == bn && stages == st)                                                            \
        return p.tma ? launch_one<bn, st, KIND_BF16_TMA, 8>(p, map, ymap, grid, stream)              \
                     : launch_one<bn, st, KIND_BF16_CPASYNC, 8>(p, map, ymap, grid, stream);
    TC_BF16_CONFIGS(X)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace convfwd
