// Backward weight of the grouped convolution on the tensor cores (bf16 in, fp32 accumulate):
// the "bwd_weight" variant that page "composable_kernel dispatcher/heuristics/
// LEARNINGS_GROUPED_CONV.md", section 6, names for the NHWGC / GKYXC / NHWGK layouts.
//
//   dw[g][k][tap][c] = sum over output pixels m of x[source(m, tap)][g][c] * dy[m][g][k]
//
// Per group this is a GEMM whose reduction runs over output pixels.  Both operands are read
// in the layouts they already have: a TMA box of 64 channels x 64 pixels (128-byte rows, one
// pixel per row, 128-byte swizzle) is, for the MMA, an MN-major tile whose MN index is the
// channel and whose K index is the pixel, so no transpose is ever materialised:
//   A (rows of D): x at the pixels one tap reads, two 64-channel halves (tap, channel block)
//                  per 128-row tile, 8 KB apart (the descriptor's MN-block stride);
//   B (columns):   dy at the output pixels, BN/64 blocks of 64 output channels, 8 KB apart.
// 8-pixel groups are 1 KB apart (the descriptor's K-group stride); each MMA consumes 16
// pixels (2 KB of each tile).  Padding, the stride and the ragged end of a row come from the
// TMA box: out-of-range pixels read as zero, and the conv stride is the box's element stride
// along W.  Channels beyond C or K only feed accumulator rows / columns that are never stored.
//
// Roles (192 threads): warp 0 lane 0 issues the TMA loads into a ring of stages (each stage
// holds CH chunks of 64 pixels); warp 1 issues the MMAs (elect.sync) and commits once per
// stage; warps 2-5 (one per TMEM lane quarter) read the accumulator and store dw, or fp32
// partial sums when the pixels are split across CTAs.  Every wait is bounded: on timeout the
// kernel raises the error word and returns after releasing its tensor memory.
#include <cuda.h>

#include "tc_common.cuh"

namespace convfwd {
namespace {

constexpr int WG_THREADS = 192;
constexpr uint32_t HALF_BYTES = 64 * 128;   // one box: 64 pixels x 64 channels of bf16

// PL: bf16 planes per operand.  1 for bf16 I/O; 3 for fp32 I/O, whose x and dy arrive split
// into hi + mid + lo bf16 planes (each the bf16 rounding of what the planes before it leave, so
// the three sum to the fp32 value within 2^-24 of it); the tile then accumulates the six
// products hi*hi, hi*mid, mid*hi, hi*lo, lo*hi, mid*mid (the dropped ones are below 2^-22 of
// |x dy|), in fp32, and dw is stored in fp32.
template <int BN, int CH, int PL>
struct WgCfg {
    static constexpr uint32_t A_PLANE = 2 * HALF_BYTES;             // two channel halves
    static constexpr uint32_t B_PLANE = (BN / 64) * HALF_BYTES;     // BN/64 channel blocks of dy
    static constexpr uint32_t A_CHUNK = PL * A_PLANE;
    static constexpr uint32_t B_CHUNK = PL * B_PLANE;
    static constexpr uint32_t CHUNK = A_CHUNK + B_CHUNK;
    static constexpr uint32_t STAGE = CH * CHUNK;
    static constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
};

// Shared-memory matrix descriptor of an MN-major operand, 128-byte swizzle: 64-element MN
// blocks mn_stride bytes apart (leading byte offset), 8-row K groups 1 KB apart (stride byte
// offset).
__device__ __forceinline__ uint64_t sw128_mn_desc(uint32_t saddr, uint32_t mn_stride) {
    uint64_t d = (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((mn_stride >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

struct ChunkPos {
    int n, od, oh, ow0;
};

__device__ __forceinline__ ChunkPos chunk_pos(const WgradTcParams& p, int q) {
    const Geom& g = p.g;
    ChunkPos c;
    const int wb = q % p.nwb;
    int r = q / p.nwb;
    c.oh = r % g.Ho;
    r /= g.Ho;
    c.od = r % g.Do;
    c.n = r / g.Do;
    c.ow0 = wb * 64;
    return c;
}

template <int BN, int CH, int STAGES, int PL>
__global__ void __launch_bounds__(WG_THREADS, 1)
    conv_wgrad_tc_kernel(const __grid_constant__ WgradTcParams p, const __grid_constant__ CUtensorMap xmap,
                         const __grid_constant__ CUtensorMap dymap) {
    using W = WgCfg<BN, CH, PL>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const uint32_t bar0 = sbase + STAGES * W::STAGE;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (STAGES + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * STAGES);
    uint8_t* misc = smem + (bar0 + 8u * (2 * STAGES + 1) - sbase);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Geom& g = p.g;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), W::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (p.pdl) {   // the next kernel may start its set-up; x and dy may come from the previous one
        griddep_launch();
        griddep_wait();
    }

    // this CTA's unit: row tile fastest, so neighbouring CTAs share their dy chunks in L2
    const int u = blockIdx.x;
    const int rt = u % p.RT;
    int r = u / p.RT;
    const int split = r % p.splits;
    r /= p.splits;
    const int nt = r % p.NT;
    const int gi = r / p.NT;        // group (pack > 1: group pack)
    const int cbase = gi * p.pack * g.C, kbase = gi * p.pack * g.K;
    const int q0 = split * p.qps;
    const int q1 = min(q0 + p.qps, p.Q);
    const int nchunks = q1 - q0;
    const int nstages = (nchunks + CH - 1) / CH;

    if (warp == 0) {
        if (lane == 0) {
            // the two channel halves of this row tile: tap and channel block, tap offsets
            int cin[2], dz[2], dyo[2], dxo[2];
            bool hv[2];
            for (int hh = 0; hh < 2; ++hh) {
                const int h = 2 * rt + hh;
                hv[hh] = h < p.halves;
                const int tap = hv[hh] ? h / p.cbh : 0;
                cin[hh] = cbase + (hv[hh] ? (h - tap * p.cbh) * 64 : 0);
                const int z = tap / (g.Y * g.X), rem = tap - z * g.Y * g.X;
                const int y = rem / g.X, x = rem - y * g.X;
                dz[hh] = z * g.dd - g.pd;
                dyo[hh] = y * g.dh - g.ph;
                dxo[hh] = x * g.dw - g.pw;
            }
            const uint32_t bytes_chunk = PL * ((hv[1] ? 2 : 1) * HALF_BYTES + W::B_PLANE);
            int issued = 0;
            for (int st = 0; st < nstages; ++st) {
                const int s = st % STAGES;
                if (st >= STAGES && !wait_bar(empty_bar(s), ((st / STAGES) - 1) & 1, abort_flag, p.err)) break;
                issued = st + 1;
                const int nc = min(CH, nchunks - st * CH);
                mbar_arrive_expect_tx(full_bar(s), nc * bytes_chunk);
                for (int c = 0; c < nc; ++c) {
                    const ChunkPos cp = chunk_pos(p, q0 + st * CH + c);
                    const uint32_t dst = sbase + s * W::STAGE + c * W::CHUNK;
                    // plane pl of image n is image pl*N + n of the plane tensors
                    for (int pl = 0; pl < PL; ++pl) {
                        const int ni = pl * g.N + cp.n;
                        for (int hh = 0; hh < 2; ++hh)
                            if (hv[hh])
                                tma_load_5d(dst + pl * W::A_PLANE + hh * HALF_BYTES, &xmap, cin[hh],
                                            cp.ow0 * g.sw + dxo[hh], cp.oh * g.sh + dyo[hh], cp.od * g.sd + dz[hh], ni,
                                            full_bar(s));
                        for (int j = 0; j < BN / 64; ++j)
                            tma_load_5d(dst + W::A_CHUNK + pl * W::B_PLANE + j * HALF_BYTES, &dymap,
                                        kbase + nt * BN + j * 64, cp.ow0, cp.oh, cp.od, ni, full_bar(s));
                    }
                }
            }
            // before the CTA can exit, the copies of the last stages issued must have landed
            // (they have unless the MMA role gave up); a bounded wait, whatever the abort flag
            const unsigned long long t0 = globaltimer();
            for (int st = issued > STAGES ? issued - STAGES : 0; st < issued; ++st)
                while (!mbar_try_wait(full_bar(st % STAGES), (st / STAGES) & 1) && globaltimer() - t0 < WAIT_LIMIT_NS) {
                }
        }
    } else if (warp == 1) {
        constexpr uint32_t IDESC = idesc_f32acc(128, BN, 1u) | (1u << 15) | (1u << 16);   // A, B MN-major
        bool ok = true;
        for (int st = 0; st < nstages && ok; ++st) {
            const int s = st % STAGES;
            ok = wait_bar_warp(full_bar(s), (st / STAGES) & 1, abort_flag, p.err);
            if (!ok) break;
            tc_fence_after();
            const int nc = min(CH, nchunks - st * CH);
            for (int c = 0; c < nc; ++c) {
                const uint32_t a = sbase + s * W::STAGE + c * W::CHUNK;
                const uint32_t b = a + W::A_CHUNK;
                // plane pairs (A, B): hi*hi only, or the six that carry fp32 accuracy
                constexpr int NP = PL == 1 ? 1 : 6;
                constexpr int PA[6] = {0, 0, 1, 0, 2, 1}, PB[6] = {0, 1, 0, 2, 0, 1};
                // plane and K-step offsets move only the descriptors' start-address field
                const uint64_t da = sw128_mn_desc(a, HALF_BYTES), db = sw128_mn_desc(b, HALF_BYTES);
#pragma unroll
                for (int k = 0; k < 4; ++k)
#pragma unroll
                    for (int q = 0; q < NP; ++q)
                        mma_bf16_warp(tmem, da + (uint64_t)((PA[q] * W::A_PLANE + k * 2048) >> 4),
                                      db + (uint64_t)((PB[q] * W::B_PLANE + k * 2048) >> 4), IDESC,
                                      (st > 0 || c > 0 || k > 0 || q > 0) ? 1u : 0u);
            }
            mma_commit_warp(empty_bar(s));
        }
        if (ok) mma_commit_warp(done_bar);
    } else {
        // epilogue: TMEM lane quarter (warp % 4); row -> (half, channel) -> (tap, c)
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const int h = 2 * rt + (row >> 6);
        const int tap = h / p.cbh;
        // packed groups: row (row & 63) is channel c of group a of the pack, and only the
        // columns of the same group (a*K .. a*K + K-1) belong to it
        const int a = p.pack > 1 ? (row & 63) / g.C : 0;
        const int c = p.pack > 1 ? (row & 63) - a * g.C : (h - tap * p.cbh) * 64 + (row & 63);
        const int grp = gi * p.pack + a;
        const bool row_ok = h < p.halves && c < g.C && a < p.pack && grp < g.G;
        const bool ok = wait_bar_warp(done_bar, 0, abort_flag, p.err, true);
        if (ok) {
            tc_fence_after();
            const int NJ = g.taps * g.C;
            const long long col0 = (long long)tap * g.C + c;
            const uint32_t taddr = tmem + ((uint32_t)(wq * 32) << 16);
            for (int cb = 0; cb < BN; cb += 16) {
                const int k0 = nt * BN + cb;
                if (k0 >= p.pack * g.K) break;   // warp-uniform
                uint32_t v[16];
                __syncwarp();
                tmem_ld16(taddr + (uint32_t)cb, v);
                tmem_ld_wait();
                if (!row_ok) continue;
                if (p.pack == 1) {
                    // columns k0 .. k0+15 (those below K) of row (tap, c): element e at offset
                    // e * NJ from the first; the warp's 32 rows are 32 consecutive c
                    const int ne = g.K - k0 < 16 ? g.K - k0 : 16;
                    const long long o0 = ((long long)grp * g.K + k0) * NJ + col0;
                    if (p.splits > 1 || PL == 3) {
                        float* w = (p.splits > 1 ? p.ws + (long long)split * g.G * g.K * NJ
                                                 : reinterpret_cast<float*>(p.dw)) + o0;
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (e < ne) w[e * NJ] = __uint_as_float(v[e]);
                    } else {
                        __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(p.dw) + o0;
#pragma unroll
                        for (int e = 0; e < 16; ++e)
                            if (e < ne) w[e * NJ] = __float2bfloat16_rn(__uint_as_float(v[e]));
                    }
                    continue;
                }
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    int k = k0 + e;
                    {   // packed groups: column -> (group of the pack, channel); keep the diagonal block
                        const int b = k / g.K;
                        if (b != a) continue;
                        k -= b * g.K;
                    }
                    const long long o = ((long long)grp * g.K + k) * NJ + col0;
                    const float f = __uint_as_float(v[e]);
                    if (p.splits > 1)
                        p.ws[(long long)split * g.G * g.K * NJ + o] = f;
                    else if (PL == 3)
                        reinterpret_cast<float*>(p.dw)[o] = f;
                    else
                        reinterpret_cast<__nv_bfloat16*>(p.dw)[o] = __float2bfloat16_rn(f);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, W::TMEM_COLS);
    }
}

// ---- slab mode (bf16, unit stride along W) ----
// A unit is (group or group pack, N tile, pixel split, filter plane z); its p.na accumulators
// hold every half of plane z: accumulator a the halves 2a and 2a + 1, half h = (y*X + x)*cbh + cb.
// Per chunk of 64 output pixels a stage holds one x box per (filter row y, channel block cb),
// 64 + (X-1)*dw pixels from column ow0 - pw, so tap (y, x) is the window x*dw pixel rows into
// box (y, cb) (MN-major windows start at any 128-byte row: the MMA applies the swizzle by
// absolute address, as the TMA did), plus the dy boxes, shared by every accumulator.  The two
// halves of an accumulator are two MN blocks one descriptor stride apart, whatever boxes and
// offsets they come from.
constexpr int WG_SLAB_MAX_STAGES = 8;
constexpr int WG_SLAB_MAX_NA = 8;

__global__ void __launch_bounds__(WG_THREADS, 1)
    conv_wgrad_slab_kernel(const __grid_constant__ WgradTcParams p, const __grid_constant__ CUtensorMap xmap,
                           const __grid_constant__ CUtensorMap dymap) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sbase = (raw + 1023u) & ~1023u;
    uint8_t* smem = smem_raw + (sbase - raw);
    const int S = p.stages;
    const uint32_t stage_bytes = (uint32_t)p.stage_bytes;
    const uint32_t bar0 = sbase + (uint32_t)S * stage_bytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (WG_SLAB_MAX_STAGES + s); };
    const uint32_t done_bar = bar0 + 8u * (2 * WG_SLAB_MAX_STAGES);
    uint8_t* misc = smem + (done_bar + 8u - sbase);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(misc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(misc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const Geom& g = p.g;
    const int BN = p.BN;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        mbar_init(done_bar, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), (uint32_t)p.tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    if (p.pdl) {
        griddep_launch();
        griddep_wait();
    }

    // unit: filter plane fastest (the planes of one pixel range share their dy chunks in L2)
    const int u = blockIdx.x;
    const int z = u % g.Z;
    int r = u / g.Z;
    const int split = r % p.splits;
    r /= p.splits;
    const int nt = r % p.NT;
    const int gi = r / p.NT;
    const int cbase = gi * p.pack * g.C, kbase = gi * p.pack * g.K;
    const int q0 = split * p.qps;
    const int q1 = min(q0 + p.qps, p.Q);
    const int nchunks = q1 - q0;
    const uint32_t dy_off = (uint32_t)(p.nbox * p.box_bytes);

    if (warp == 0) {
        if (lane == 0) {
            const uint32_t tx = (uint32_t)p.nbox * (uint32_t)p.box_rows * 128u + (uint32_t)(BN / 64) * HALF_BYTES;
            int issued = 0;
            bool aborted = false;
            for (int st = 0; st < nchunks; ++st) {
                const int s = st % S;
                if (st >= S && !wait_bar(empty_bar(s), ((st / S) - 1) & 1, abort_flag, p.err)) {
                    aborted = true;
                    break;
                }
                issued = st + 1;
                mbar_arrive_expect_tx(full_bar(s), tx);
                const ChunkPos cp = chunk_pos(p, q0 + st);
                const uint32_t dst = sbase + (uint32_t)s * stage_bytes;
                const int dd = cp.od * g.sd - g.pd + z * g.dd;
                for (int b = 0; b < p.nbox; ++b) {
                    const int y = b / p.cbh, cb = b - y * p.cbh;
                    tma_load_5d(dst + (uint32_t)(b * p.box_bytes), &xmap, cbase + cb * 64, cp.ow0 - g.pw,
                                cp.oh * g.sh - g.ph + y * g.dh, dd, cp.n, full_bar(s));
                }
                for (int j = 0; j < BN / 64; ++j)
                    tma_load_5d(dst + dy_off + (uint32_t)j * HALF_BYTES, &dymap, kbase + nt * BN + j * 64, cp.ow0, cp.oh,
                                cp.od, cp.n, full_bar(s));
            }
            (void)aborted;
            // the copies of the last stages issued must have landed before the CTA exits
            const unsigned long long t0 = globaltimer();
            for (int st = issued > S ? issued - S : 0; st < issued; ++st)
                while (!mbar_try_wait(full_bar(st % S), (st / S) & 1) && globaltimer() - t0 < WAIT_LIMIT_NS) {
                }
        }
    } else if (warp == 1) {
        const uint32_t IDESC = idesc_f32acc(128, BN, 1u) | (1u << 15) | (1u << 16);   // A, B MN-major
        // per accumulator: its first half's window (bytes into a stage) and the distance to the second
        uint32_t aoff[WG_SLAB_MAX_NA], albo[WG_SLAB_MAX_NA];
#pragma unroll
        for (int a = 0; a < WG_SLAB_MAX_NA; ++a) {
            aoff[a] = albo[a] = 0;
            if (a < p.na) {
                uint32_t o[2];
                for (int hh = 0; hh < 2; ++hh) {
                    const int h = min(2 * a + hh, p.hpp - 1);   // a missing second half repeats the first
                    const int t = h / p.cbh, cb = h - t * p.cbh;
                    const int y = t / g.X, x = t - y * g.X;
                    o[hh] = (uint32_t)((y * p.cbh + cb) * p.box_bytes + x * g.dw * 128);
                }
                aoff[a] = o[0];
                albo[a] = o[1] - o[0];
            }
        }
        // Descriptors of stage 0 built once; a stage, a K step (2048 bytes) and the stage
        // offset move only the start-address field (address / 16, 14 bits: no carry within
        // shared memory), so the issue loop adds to them instead of rebuilding them (measured:
        // building every descriptor in the loop left the MMA thread at ~120 cycles per MMA).
        uint64_t ad0[WG_SLAB_MAX_NA];
#pragma unroll
        for (int a = 0; a < WG_SLAB_MAX_NA; ++a) ad0[a] = sw128_mn_desc(sbase + aoff[a], albo[a]);
        const uint64_t bd0 = sw128_mn_desc(sbase + dy_off, HALF_BYTES);
        bool ok = true;
        for (int st = 0; st < nchunks && ok; ++st) {
            const int s = st % S;
            ok = wait_bar_warp(full_bar(s), (st / S) & 1, abort_flag, p.err);
            if (!ok) break;
            tc_fence_after();
            const uint64_t sd = (uint64_t)(((uint32_t)s * stage_bytes) >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint64_t kd = sd + (uint64_t)(k * (2048 >> 4));
                const uint64_t bd = bd0 + kd;
#pragma unroll
                for (int a = 0; a < WG_SLAB_MAX_NA; ++a)
                    if (a < p.na)
                        mma_bf16_warp(tmem + (uint32_t)(a * BN), ad0[a] + kd, bd, IDESC, (st > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit_warp(empty_bar(s));
        }
        if (ok) mma_commit_warp(done_bar);
    } else {
        // epilogue: TMEM lane quarter (warp % 4); per accumulator a, row -> half -> (tap, c)
        const int wq = warp & 3;
        const int row = wq * 32 + lane;
        const bool ok = wait_bar_warp(done_bar, 0, abort_flag, p.err, true);
        if (ok) {
            tc_fence_after();
            const int NJ = g.taps * g.C;
            const int pa = p.pack > 1 ? (row & 63) / g.C : 0;
            const int grp = gi * p.pack + pa;
            for (int a = 0; a < p.na; ++a) {
                const int h = 2 * a + (row >> 6);
                const int t = h / p.cbh;
                const int c = p.pack > 1 ? (row & 63) - pa * g.C : (h - t * p.cbh) * 64 + (row & 63);
                const int tap = z * g.Y * g.X + t;
                const bool row_ok = h < p.hpp && c < g.C && pa < p.pack && grp < g.G;
                const long long col0 = (long long)tap * g.C + c;
                const uint32_t taddr = tmem + ((uint32_t)(wq * 32) << 16) + (uint32_t)(a * BN);
                for (int cb = 0; cb < BN; cb += 16) {
                    const int k0 = nt * BN + cb;
                    if (k0 >= p.pack * g.K) break;   // warp-uniform
                    uint32_t v[16];
                    __syncwarp();
                    tmem_ld16(taddr + (uint32_t)cb, v);
                    tmem_ld_wait();
                    if (!row_ok) continue;
                    if (p.pack == 1) {
                        // columns k0 .. k0+15 (those below K) of row (tap, c): element e at
                        // offset e * NJ from the first; the warp's 32 rows are 32 consecutive c
                        const int ne = g.K - k0 < 16 ? g.K - k0 : 16;
                        const long long o0 = ((long long)grp * g.K + k0) * NJ + col0;
                        if (p.splits > 1) {
                            float* w = p.ws + (long long)split * g.G * g.K * NJ + o0;
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                if (e < ne) w[e * NJ] = __uint_as_float(v[e]);
                        } else {
                            __nv_bfloat16* w = reinterpret_cast<__nv_bfloat16*>(p.dw) + o0;
#pragma unroll
                            for (int e = 0; e < 16; ++e)
                                if (e < ne) w[e * NJ] = __float2bfloat16_rn(__uint_as_float(v[e]));
                        }
                        continue;
                    }
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        int k = k0 + e;
                        const int b = k / g.K;   // packed groups: keep the diagonal block
                        if (b != pa) continue;
                        k -= b * g.K;
                        const long long o = ((long long)grp * g.K + k) * NJ + col0;
                        const float f = __uint_as_float(v[e]);
                        if (p.splits > 1)
                            p.ws[(long long)split * g.G * g.K * NJ + o] = f;
                        else
                            reinterpret_cast<__nv_bfloat16*>(p.dw)[o] = __float2bfloat16_rn(f);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
    }
}

template <int BN, int CH, int STAGES, int PL>
constexpr size_t wg_smem_bytes() {
    return 1024 + (size_t)STAGES * WgCfg<BN, CH, PL>::STAGE + 8 * (2 * STAGES + 1) + 16;
}

template <int BN, int CH, int STAGES, int PL>
cudaError_t launch_wg(const WgradTcParams& p, const CUtensorMap& xmap, const CUtensorMap& dymap, cudaStream_t stream) {
    auto kern = conv_wgrad_tc_kernel<BN, CH, STAGES, PL>;
    constexpr size_t smem = wg_smem_bytes<BN, CH, STAGES, PL>();
    static_assert(smem <= 232448, "shared memory budget");
    static bool attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    return launch_kernel(kern, dim3(p.total_units), dim3(WG_THREADS), smem, stream, p.pdl != 0, 1, p, xmap, dymap);
}

}  // namespace

cudaError_t launch_wgrad_tc(const WgradTcParams& p, const CUtensorMap* xmap, const CUtensorMap* dymap,
                            cudaStream_t stream) {
    if (p.slab) {
        const size_t smem = 1024 + (size_t)p.stages * p.stage_bytes + 8 * (2 * WG_SLAB_MAX_STAGES + 1) + 16;
        if (p.stages < 2 || p.stages > WG_SLAB_MAX_STAGES || p.na < 1 || p.na > WG_SLAB_MAX_NA || smem > 232448 ||
            p.na * p.BN > p.tmem_cols || p.tmem_cols > 512 || p.planes != 1)
            return cudaErrorInvalidValue;
        static bool attr_set[64];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64 || !attr_set[dev]) {
            e = cudaFuncSetAttribute(conv_wgrad_slab_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
            if (e != cudaSuccess) return e;
            if (dev >= 0 && dev < 64) attr_set[dev] = true;
        }
        return launch_kernel(conv_wgrad_slab_kernel, dim3(p.total_units), dim3(WG_THREADS), smem, stream, p.pdl != 0, 1,
                             p, *xmap, *dymap);
    }
    if (p.planes == 3) {
        switch (p.BN) {
            case 64: return launch_wg<64, 1, 3, 3>(p, *xmap, *dymap, stream);
            case 128: return launch_wg<128, 1, 2, 3>(p, *xmap, *dymap, stream);
        }
        return cudaErrorInvalidValue;
    }
    switch (p.BN) {
        case 64: return launch_wg<64, 2, 4, 1>(p, *xmap, *dymap, stream);
        case 128: return launch_wg<128, 2, 3, 1>(p, *xmap, *dymap, stream);
        case 256: return launch_wg<256, 1, 4, 1>(p, *xmap, *dymap, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace convfwd
