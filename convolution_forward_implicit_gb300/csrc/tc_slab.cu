// Slab mode of the tensor-core implicit GEMM, for convolutions with stride 1: one TMA box
// per (output tile, input plane, channel block) brings the input rows the whole tile needs
// (the tile's rows plus the filter's reach), and every tap of that plane reads the box as a
// row-shifted window through the MMA's shared-memory descriptor.  The same input bytes serve
// Y*X taps, where the per-tap mode copies them once per tap.
//
// Layout.  An output tile is BH rows x BW columns of one output plane.  The slab holds
// HR = BH + dh*(Y-1) input rows of BWs = BW + dw*(X-1) pixels each, starting at input column
// ow0 - pw, each pixel one 128-byte row of channels (64 bf16 or 32 fp32), 128-byte swizzled
// by the TMA.  Accumulator row r stands for output pixel (oh0 + r / BWs, ow0 + r % BWs): with
// the slab's row pitch BWs, tap (y, x) is the 128-row window starting at slab row
// y*dh*BWs + x*dw.  Rows whose column r % BWs lands past BW are computed and discarded.
// Windows start at arbitrary 128-byte rows.  The tensor core takes the swizzle phase of a
// row from its absolute shared-memory address, as the TMA did when it wrote the row, so a
// window's descriptor is the plain one at its start address, with the matrix base offset
// field left 0 (measured: setting it to the start's phase corrupts every window that is
// not 1024-byte aligned).
//
// Roles (warps): 0-7 epilogue (as in the per-tap kernel), 8 slab copies, 9-11 weight copies
// (X taps' weight tiles in one bulk copy; ring stage s owned by warp 9 + s % 3), 12 MMA
// issue (with tile pairs, 12 and 13: one issuer per accumulator), then (3xTF32 only) 4 warps
// for the hi/lo split of each slab.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"
#include "tc_common.cuh"

namespace convfwd {
namespace {

constexpr int SLAB_MAX_SA = 4;
constexpr int SLAB_MAX_SB = 8;

// NMMA MMA-issuing warps.  An N = 64 MMA (128x64x16) runs in ~48 cycles, while one thread
// issues one only every ~75 cycles (its descriptors, the elect and the issue itself; measured:
// MMAs of half the width, same count, took within 8% of the time): the kernel was bound by
// issue.  With tile pairs, each accumulator gets its own issuer; the stages both read and the
// accumulator-full barrier then take one commit from each.
template <bool TF32, int NMMA>
struct SlabRoles {
    static constexpr int A_WARP = EPI_WARPS;
    static constexpr int B_WARP0 = EPI_WARPS + 1;
    static constexpr int B_WARPS = 3;
    static constexpr int MMA_WARP = EPI_WARPS + 4;
    static constexpr int CVT_WARP0 = MMA_WARP + NMMA;
    static constexpr int CVT_WARPS = TF32 ? 4 : 0;
    static constexpr int THREADS = (CVT_WARP0 + CVT_WARPS) * 32;
};

// BY, BT: filter rows Y (weight stages per k-group) and columns X (taps per stage) fixed at
// compile time for the common 3x3 and 1x3 filters, so the MMA issue loop over a k-group's taps
// unrolls with constant descriptor offsets; 0 reads them from the parameters.  Measured on
// 3x3 filters: the unrolled issue loop makes the whole kernel 1.2x (2D) to 1.3x (3D) faster.
//
// NACC: accumulators per unit.  With 2 (tile pairs), a unit is two output tiles stacked along
// H that share one slab (their halo rows once) and one pass over the weights: every tap issues
// its MMAs into both accumulators from windows slab_pair_rows apart, against the same weight
// tile.  The per-unit waits, commits and copies then serve twice the MMAs.
//
// PLAIN: compiled for layers with no bias and no activation (the bias and GELU code left out:
// 2D grouped layers 1.6% faster).
template <int BN, bool TF32, int BY, int BT, int NACC, bool PLAIN = false>
__global__ void __launch_bounds__(SlabRoles<TF32, (TF32 ? 1 : NACC)>::THREADS, 1)
    conv_fwd_slab_kernel(const __grid_constant__ TcParams p, const __grid_constant__ CUtensorMap act_map) {
    constexpr int NMMA = TF32 ? 1 : NACC;          // MMA-issuing warps (one per accumulator of a unit)
    using R = SlabRoles<TF32, NMMA>;
    constexpr uint32_t B_TILE = BN * 128;
    constexpr uint32_t TMEM_COLS = (2 * NACC * BN < 32) ? 32 : 2 * NACC * BN;   // 2 buffers of NACC accumulators
    const int SA = p.slab_sa, SB = p.slab_sb;
    const uint32_t a_stage = (uint32_t)p.slab_a_stage;           // TF32: hi half, then lo half
    const uint32_t a_half = TF32 ? a_stage / 2 : a_stage;
    const uint32_t b_tap = TF32 ? 2 * B_TILE : B_TILE;            // one tap's weights (TF32: hi, lo)
    const uint32_t b_stage = (uint32_t)p.slab_btaps * b_tap;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const uint32_t sA = sbase;
    const uint32_t sB = sA + SA * a_stage;
    const uint32_t stg_off = SA * a_stage + SB * b_stage;
    // each epilogue warp stages one chunk of its BN/2 columns: 32 rows x (BN/2 x element size)
    constexpr uint32_t STG_W = stg_warp_bytes<(BN / 2 < 16 ? 16 : BN / 2), (TF32 ? 4 : 2)>();
    const uint32_t bar0 = sbase + stg_off + EPI_WARPS * STG_W;
    auto full_a = [&](int s) { return bar0 + 8u * s; };
    auto empty_a = [&](int s) { return bar0 + 8u * (SLAB_MAX_SA + s); };
    auto cvt_a = [&](int s) { return bar0 + 8u * (2 * SLAB_MAX_SA + s); };
    auto full_b = [&](int s) { return bar0 + 8u * (3 * SLAB_MAX_SA + s); };
    auto empty_b = [&](int s) { return bar0 + 8u * (3 * SLAB_MAX_SA + SLAB_MAX_SB + s); };
    const uint32_t bar_t = bar0 + 8u * (3 * SLAB_MAX_SA + 2 * SLAB_MAX_SB);
    auto tfull_bar = [&](int a) { return bar_t + 8u * a; };
    auto tempty_bar = [&](int a) { return bar_t + 8u * (2 + a); };
    auto drain_bar = [&](int mw) { return bar_t + 8u * (4 + mw); };   // one per MMA warp
    uint8_t* misc = smem + (bar_t + 8u * 6 - sbase);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < SA; ++s) {
            mbar_init(full_a(s), 1);
            mbar_init(empty_a(s), NMMA);
            mbar_init(cvt_a(s), R::CVT_WARPS > 0 ? R::CVT_WARPS : 1);
        }
        if (p.slab_resident) {
            mbar_init(full_b(0), R::B_WARPS);
            mbar_init(empty_b(0), NMMA);
        } else {
            for (int s = 0; s < SB; ++s) {
                mbar_init(full_b(s), 1);
                mbar_init(empty_b(s), NMMA);
            }
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull_bar(a), NMMA);
            mbar_init(tempty_bar(a), EPI_WARPS);
        }
        for (int mw = 0; mw < NMMA; ++mw) mbar_init(drain_bar(mw), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        fence_proxy_async();
    }
    if (warp == R::A_WARP && lane == 0)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&act_map)) : "memory");
    if (warp == R::MMA_WARP) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // set up: the next kernel on the stream may start (its own set-up and weight loads)
    if (p.pdl) griddep_launch();

    const Geom& g = p.g;
    const int cblk = TF32 ? 32 : 64;
    const int nbg = BY > 0 ? BY : p.slab_nbg;        // weight stages per k-group (filter rows)
    const int btaps = BT > 0 ? BT : p.slab_btaps;   // taps per weight stage (filter columns)

    if (warp == R::A_WARP) {
        // ------------------------------------------------------------ slab copies
        if (lane == 0) {
            if (p.pdl && (int)blockIdx.x < p.total_units) {
                // the first unit's first slabs go into L2 while the previous kernel finishes
                int mt, gi, nt, split;
                decode_unit(p, blockIdx.x, mt, gi, nt, split);
                const TileOrigin to = tile_origin(p, mt);
                for (int kg = 0; kg < p.slab_nkg && kg < SA; ++kg) {
                    const int zz = fdiv(kg, p.f_cbt), cb = kg - zz * p.cbt;
                    if (p.map_kind == 0)
                        tma_prefetch_5d(&act_map, gi * g.C + cb * cblk, to.ow0 - g.pw, to.oh0 - g.ph,
                                        to.od - g.pd + zz * g.dd, to.n);
                    else
                        tma_prefetch_5d(&act_map, cb * cblk, gi, to.ow0 - g.pw, to.oh0 - g.ph, to.n);
                }
            }
            if (p.pdl) griddep_wait();   // x may come from the previous kernel on the stream
            const uint32_t a_tx = (uint32_t)(p.slab_hr * p.slab_bws) * 128u;
            Ring ra(SA);
            bool aborted = false;
            for (int u = blockIdx.x; u < p.total_units && !aborted; u += gridDim.x) {
                int mt, gi, nt, split;
                decode_unit(p, u, mt, gi, nt, split);
                const TileOrigin to = tile_origin(p, mt);
                const int w0 = to.ow0 - g.pw, h0 = to.oh0 - g.ph;
                for (int kg = 0; kg < p.slab_nkg; ++kg, ra.next()) {
                    const int zz = fdiv(kg, p.f_cbt), cb = kg - zz * p.cbt;
                    const int s = ra.s;
                    const uint32_t ph = ra.ph;
                    if (!wait_bar(empty_a(s), ph ^ 1u, abort_flag, p.err, p.sleep_mask & 1)) { aborted = true; break; }
                    mbar_arrive_expect_tx(full_a(s), a_tx);
                    if (p.map_kind == 0)
                        tma_load_5d(sA + s * a_stage, &act_map, gi * g.C + cb * cblk, w0, h0,
                                    to.od - g.pd + zz * g.dd, to.n, full_a(s));
                    else
                        tma_load_5d(sA + s * a_stage, &act_map, cb * cblk, gi, w0, h0, to.n, full_a(s));
                }
            }
        }
        __syncwarp();
    } else if (warp >= R::B_WARP0 && warp < R::B_WARP0 + R::B_WARPS) {
        // ------------------------------------------------------------ weight copies
        if (lane == 0) {
            const uint8_t* wp = reinterpret_cast<const uint8_t*>(p.wpack);
            const int bw = warp - R::B_WARP0;
            const int nchunk = p.slab_nkg * nbg;    // chunks of btaps taps, in slab order
            bool aborted = false;
            if (p.slab_resident) {
                // The whole weight set of the current (group, N tile) stays in shared memory;
                // it is reloaded only when the next unit changes group or N tile.  Each copy
                // warp brings every third chunk; all three arrive on the one full barrier.
                int prev = -1;
                uint32_t j = 0;
                for (int u = blockIdx.x; u < p.total_units && !aborted; u += gridDim.x) {
                    int mt, gi, nt, split;
                    decode_unit(p, u, mt, gi, nt, split);
                    const int key = gi * p.num_nt + nt;
                    if (key == prev) continue;
                    prev = key;
                    // only the first weight set loads before the previous kernel has completed;
                    // a wait that can block (and time out) comes after it
                    if (p.pdl && j == 1) griddep_wait();
                    if (!wait_bar(empty_b(0), (j & 1u) ^ 1u, abort_flag, p.err, p.sleep_mask & 1)) {
                        aborted = true;
                        break;
                    }
                    const int mine = nchunk > bw ? (nchunk - bw + R::B_WARPS - 1) / R::B_WARPS : 0;
                    mbar_arrive_expect_tx(full_b(0), (uint32_t)mine * b_stage);
                    const size_t base = (size_t)key * p.nkb * b_tap;
                    for (int c = bw; c < nchunk; c += R::B_WARPS)
                        bulk_g2s(sB + c * b_stage, wp + base + (size_t)c * b_stage, b_stage, full_b(0));
                    ++j;
                }
            } else {
                uint32_t ib = 0;
                Ring rb(SB);
                bool waited = false;
                for (int u = blockIdx.x; u < p.total_units && !aborted; u += gridDim.x) {
                    int mt, gi, nt, split;
                    decode_unit(p, u, mt, gi, nt, split);
                    for (int c = 0; c < nchunk; ++c, ++ib, rb.next()) {
                        const int s = rb.s;
                        if (s % R::B_WARPS != bw) continue;    // each ring stage has one owner warp
                        const uint32_t ph = rb.ph;
                        // the first pass over the ring loads before the previous kernel has
                        // completed; waits that can block (and time out) come after it
                        if (p.pdl && ib >= (uint32_t)SB && !waited) {
                            griddep_wait();
                            waited = true;
                        }
                        if (!wait_bar(empty_b(s), ph ^ 1u, abort_flag, p.err, p.sleep_mask & 1)) {
                            aborted = true;
                            break;
                        }
                        mbar_arrive_expect_tx(full_b(s), b_stage);
                        // chunk c = kg*nbg + bg holds K blocks c*btaps .. c*btaps + btaps-1
                        const size_t off = ((size_t)(gi * p.num_nt + nt) * p.nkb + (size_t)c * btaps) * b_tap;
                        bulk_g2s(sB + s * b_stage, wp + off, b_stage, full_b(s));
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp >= R::MMA_WARP && warp < R::MMA_WARP + NMMA) {
        // ------------------------------------------------------------ MMA issue (whole warp)
        // issuer mw takes accumulator mw of each unit (with NMMA = 1, all of them); every issuer
        // waits for the same stages and commits each release once
        const int mw = warp - R::MMA_WARP;
        // bounded waits start once the previous kernel on the stream has completed
        if (p.pdl) griddep_wait();
        constexpr uint32_t IDESC = idesc_f32acc(BM, BN, TF32 ? 2u : 1u);
        const bool msleep = (p.sleep_mask & 4) != 0;
        const bool resident = p.slab_resident != 0;
        // weight set of unit u: (group, N tile) = u mod KT (slab plans do not split K); from one
        // unit of this CTA to its next the key advances by gridDim.x mod KT
        const int KT = p.g.G * p.num_nt;
        const int kstep = (int)(gridDim.x % (unsigned)KT);
        int key = (int)(blockIdx.x % (unsigned)KT);
        Ring ra(SA), rb(SB);
        uint32_t tile_i = 0, jw = 0;
        int prev = -1;
        bool aborted = false;
        for (int u = blockIdx.x; u < p.total_units && !aborted; u += gridDim.x, ++tile_i) {
            const int acc = tile_i & 1;
            const uint32_t aph = (tile_i >> 1) & 1u;
            int next_key = key + kstep;
            if (next_key >= KT) next_key -= KT;
            if (u + (int)gridDim.x >= p.total_units) next_key = -1;
            if (!wait_bar_warp(tempty_bar(acc), aph ^ 1u, abort_flag, p.err, msleep)) {
                aborted = true;
                break;
            }
            if (resident) {
                if (key != prev) {
                    if (!wait_bar_warp(full_b(0), jw & 1u, abort_flag, p.err, msleep)) {
                        aborted = true;
                        break;
                    }
                    ++jw;
                    prev = key;
                }
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + (uint32_t)(acc * NACC * BN);
            uint32_t first = 1;
            for (int kg = 0; kg < p.slab_nkg && !aborted; ++kg, ra.next()) {
                const int sa = ra.s;
                const uint32_t pha = ra.ph;
                if (!wait_bar_warp(TF32 ? cvt_a(sa) : full_a(sa), pha, abort_flag, p.err, msleep)) {
                    aborted = true;
                    break;
                }
                tc_fence_after();
                const uint32_t a0 = sA + sa * a_stage;
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
                        const uint64_t bd = sw128_desc(b0 + t * b_tap);
#pragma unroll
                        for (int j = 0; j < NACC; ++j) {
                            if (NMMA > 1 && j != mw) continue;
                            const uint32_t a_addr = a0 + (row + (uint32_t)(j * p.slab_pair_rows)) * 128u;
                            const uint64_t ad = sw128_desc(a_addr);
                            const uint32_t dj = d_tmem + (uint32_t)(j * BN);
                            if (TF32) {
                                const uint64_t alo = sw128_desc(a_addr + a_half);
                                const uint64_t blo = bd + (B_TILE >> 4);
#pragma unroll
                                for (int k = 0; k < 4; ++k) {
                                    mma_tf32_warp(dj, alo + 2u * k, bd + 2u * k, IDESC, (first && k == 0) ? 0u : 1u);
                                    mma_tf32_warp(dj, ad + 2u * k, blo + 2u * k, IDESC, 1u);
                                    mma_tf32_warp(dj, ad + 2u * k, bd + 2u * k, IDESC, 1u);
                                }
                            } else {
#pragma unroll
                                for (int k = 0; k < 4; ++k)
                                    mma_bf16_warp(dj, ad + 2u * k, bd + 2u * k, IDESC, (first && k == 0) ? 0u : 1u);
                            }
                        }
                        first = 0;
                    }
                    if (!resident) mma_commit_warp(empty_b(sb));
                }
                mma_commit_warp(empty_a(sa));
            }
            if (aborted) break;
            // the weight set is released after the last tile that uses it
            if (resident && next_key != key) mma_commit_warp(empty_b(0));
            mma_commit_warp(tfull_bar(acc));
            key = next_key;
        }
        if (aborted) {
            // wait (bounded) until every MMA issued so far has completed
            mma_commit_warp(drain_bar(mw));
            if (lane == 0) {
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(drain_bar(mw), 0) && globaltimer() - t0 < WAIT_LIMIT_NS) {}
            }
        }
        __syncwarp();
    } else if (TF32 && warp >= R::CVT_WARP0) {
        // ------------------------------------------------------------ hi/lo split (3xTF32)
        if (p.pdl) griddep_wait();
        // Every fp32 x of the slab becomes hi = x with its low 13 mantissa bits cleared (exact
        // in TF32) and lo = x - hi (exact in fp32); the MMA sums lo*w_hi + hi*w_lo + hi*w_hi.
        const int ct = threadIdx.x - R::CVT_WARP0 * 32;
        const int n16 = p.slab_hr * p.slab_bws * 8;
        Ring ra(SA);
        bool aborted = false;
        for (int u = blockIdx.x; u < p.total_units && !aborted; u += gridDim.x) {
            for (int kg = 0; kg < p.slab_nkg; ++kg, ra.next()) {
                const int s = ra.s;
                const uint32_t ph = ra.ph;
                if (!wait_bar_warp(full_a(s), ph, abort_flag, p.err)) { aborted = true; break; }
                uint4* hi = reinterpret_cast<uint4*>(smem + s * a_stage);
                uint4* lo = reinterpret_cast<uint4*>(smem + s * a_stage + a_half);
                for (int i = ct; i < n16; i += R::CVT_WARPS * 32) {
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
                if (lane == 0) mbar_arrive(cvt_a(s));
            }
        }
    } else if (warp < EPI_WARPS) {
        // ------------------------------------------------------------ epilogue
        const int wq = warp & 3;
        constexpr int SCOLS = BN / 2 < 16 ? 16 : BN / 2;   // two warps per TMEM lane quarter
        const int cb_begin = (warp >> 2) * SCOLS;
        const int cb_end = cb_begin + SCOLS < BN ? cb_begin + SCOLS : BN;
        const bool add_bias = !PLAIN && (p.epi == EPI_BIAS || p.epi == EPI_BIAS_GELU);
        const bool do_gelu = !PLAIN && (p.epi == EPI_BIAS_GELU || p.epi == EPI_GELU);
        uint8_t* stg = smem + stg_off + warp * STG_W;
        if (p.pdl) griddep_wait();   // y and bias may belong to the previous kernel
        uint32_t tile_i = 0;
        for (int u = blockIdx.x; u < p.total_units; u += gridDim.x, ++tile_i) {
            int mt, gi, nt, split;
            decode_unit(p, u, mt, gi, nt, split);
            const int acc = tile_i & 1;
            const uint32_t aph = (tile_i >> 1) & 1u;
            const TileOrigin to = tile_origin(p, mt);
            // output pixel of row rr (row pitch BWs) of accumulator j (acc_bh output rows each),
            // or -1 if it is not stored
            long long roff[NACC][EPI_MAX_LPR];
#pragma unroll
            for (int j = 0; j < NACC; ++j) {
                auto row_offset = [&](int rr) -> long long {
                    const int rh = fdiv(rr, p.f_bws), rw = rr - rh * p.slab_bws;
                    const int oh = to.oh0 + j * p.acc_bh + rh, ow = to.ow0 + rw;
                    if (rh >= p.acc_bh || rw >= p.BW || oh >= g.Ho || ow >= g.Wo) return -1;
                    return (long long)(((to.n * g.Do + to.od) * g.Ho + oh) * g.Wo + ow) * (g.G * g.K);
                };
                if (TF32) epilogue_rows<SCOLS, 4>(lane, wq, row_offset, roff[j]);
                else epilogue_rows<SCOLS, 2>(lane, wq, row_offset, roff[j]);
            }
            if (!wait_bar_warp(tfull_bar(acc), aph, abort_flag, p.err, (p.sleep_mask & 2) != 0)) break;
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < NACC; ++j) {
                const uint32_t taddr = tmem_base + ((uint32_t)(wq * 32) << 16) + (uint32_t)((acc * NACC + j) * BN);
                if (TF32)
                    epilogue_chunks<BN, SCOLS, 4>(p, taddr, lane, wq, cb_begin, cb_end, nt, gi, 0, false, add_bias,
                                                  do_gelu, stg, roff[j]);
                else
                    epilogue_chunks<BN, SCOLS, 2>(p, taddr, lane, wq, cb_begin, cb_end, nt, gi, 0, false, add_bias,
                                                  do_gelu, stg, roff[j]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == R::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int BN, bool TF32, int BY, int BT, int NACC = 1, bool PLAIN = false>
cudaError_t launch_slab_one(const TcParams& p, const CUtensorMap& map, int grid, size_t smem, cudaStream_t stream) {
    auto kern = conv_fwd_slab_kernel<BN, TF32, BY, BT, NACC, PLAIN>;
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
    return launch_kernel(kern, dim3(grid), dim3(SlabRoles<TF32, (TF32 ? 1 : NACC)>::THREADS), smem, stream,
                         p.pdl != 0, 1, p, map);
}

}  // namespace

size_t slab_smem_bytes(int BN, int tf32, int sa, int sb, size_t a_stage, int btaps) {
    const size_t b_stage = (size_t)btaps * BN * 128 * (tf32 ? 2 : 1);
    return 1024 + (size_t)sa * a_stage + (size_t)sb * b_stage + (size_t)EPI_WARPS * slab_stg_warp_bytes(BN, tf32 ? 4 : 2) +
           8 * (3 * SLAB_MAX_SA + 2 * SLAB_MAX_SB + 6) + 16;
}

cudaError_t launch_slab(const TcParams& p, const CUtensorMap* act_map, int grid, size_t smem, cudaStream_t stream) {
    if (!act_map || p.lat.on || p.slab_sa < 2 || p.slab_sa > SLAB_MAX_SA ||   // no lattice outputs here
        (!p.slab_resident && (p.slab_sb < 2 || p.slab_sb > SLAB_MAX_SB)) || smem > SLAB_SMEM_MAX)
        return cudaErrorInvalidValue;
// (3xTF32 keeps the generic loop: unrolled, its 12 MMAs per tap measured slower; tile pairs
// are bf16 only, for N tiles up to 64: wider ones run out of registers for two accumulators'
// row offsets.)
#define X(bn)                                                                                                \
    if (p.BN == bn) {                                                                                        \
        if (p.tf32) return p.slab_nacc == 1 ? launch_slab_one<bn, true, 0, 0>(p, *act_map, grid, smem, stream) \
                                             : cudaErrorInvalidValue;                                        \
        if (p.slab_nacc == 2) {                                                                              \
            if (bn > 64) return cudaErrorInvalidValue;                                                       \
            if (p.slab_btaps == 3 && p.slab_nbg == 3)                                                        \
                return p.epi == EPI_NONE                                                                     \
                           ? launch_slab_one<bn, false, 3, 3, (bn > 64 ? 1 : 2), true>(p, *act_map, grid, smem, stream) \
                           : launch_slab_one<bn, false, 3, 3, (bn > 64 ? 1 : 2)>(p, *act_map, grid, smem, stream); \
            return launch_slab_one<bn, false, 0, 0, (bn > 64 ? 1 : 2)>(p, *act_map, grid, smem, stream);    \
        }                                                                                                    \
        if (p.slab_nacc != 1) return cudaErrorInvalidValue;                                                  \
        if (p.slab_btaps == 3 && p.slab_nbg == 3) return launch_slab_one<bn, false, 3, 3>(p, *act_map, grid, smem, stream); \
        if (p.slab_btaps == 3 && p.slab_nbg == 1) return launch_slab_one<bn, false, 1, 3>(p, *act_map, grid, smem, stream); \
        return launch_slab_one<bn, false, 0, 0>(p, *act_map, grid, smem, stream);                           \
    }
    X(16) X(32) X(64) X(128) X(256)
#undef X
    return cudaErrorInvalidValue;
}

}  // namespace convfwd
