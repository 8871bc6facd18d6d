// C-ABI of the convolution-forward library: plans, weight prepacking, the forward
// dispatch, the split-K reduction and the device error word.  Declarations and the
// contract of every entry point are in include/conv.h.
#include <cuda_bf16.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <map>
#include <mutex>
#include <string>
#include <vector>
#include <new>

#include <cudaTypedefs.h>

#include "conv.h"
#include "gelu.cuh"
#include "internal.h"

using namespace convfwd;

// ----------------------------------------------------------------------------- device error word
namespace {
__device__ unsigned int g_error_word;   // bit flags raised by kernels that abandon a wait

std::mutex g_err_mu;
unsigned* g_err_ptr[64];

unsigned* error_word_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_err_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_error_word) != cudaSuccess) return nullptr;
        g_err_ptr[dev] = static_cast<unsigned*>(p);
    }
    return g_err_ptr[dev];
}

// ----------------------------------------------------------------------------- prepack kernels
// Tensor-core layout: per (group, N tile, 64-wide K block) a BN x 128-byte tile whose
// 16-byte chunk j of row n sits at chunk position j ^ (n & 7): the 128-byte swizzle the
// MMA's shared-memory descriptor expects, so the tile is copied into shared memory as is.
// K order: per_tap = 0 packs the (tap, c) chunks densely (K block kb holds chunks
// 8kb..8kb+7, crossing taps); per_tap = 1 gives every tap cbt whole 64-channel blocks
// (K block kb = tap*cbt + b holds channels 64b..64b+63 of that tap), matching one TMA box.
// Packed small groups (pack > 1): the kernel sees G/pack groups of pack*C channels and
// pack*K outputs; the packed weight of a super-group is block diagonal, output k' = jK + k
// drawing only on input channels c' = jC + c of the same original group j, zero elsewhere.
// K, C are the kernel's (packed) per-group extents, Ko, Co the caller's.
// K order 2 (slab mode) walks k-groups (input plane z, channel block b) and within each the
// Y*X taps of that plane: K block kb = ((z*cbt + b)*Y + y)*X + x.
__global__ void prepack_tc_kernel(const uint4* __restrict__ w, uint4* __restrict__ out, int K, int C, int taps,
                                  int BN, int num_nt, int nkb, int nchunks, int cpt, int per_tap, int cbt,
                                  int pack, int Ko, int Co, int Y, int X, long long total16) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total16;
         idx += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(idx & 7);
        long long r = idx >> 3;
        const int n = (int)(r % BN); r /= BN;
        const int kb = (int)(r % nkb); r /= nkb;
        const int nt = (int)(r % num_nt);
        const int g = (int)(r / num_nt);
        const int k = nt * BN + n;
        int tap, c0;
        bool ok;
        if (per_tap == 2) {
            const int kg = kb / (Y * X), t = kb - kg * (Y * X);
            const int z = kg / cbt, b = kg - z * cbt;
            tap = (z * Y + t / X) * X + t % X;
            c0 = b * 64 + j * 8;
            ok = c0 < C;
        } else if (per_tap) {
            tap = kb / cbt;
            c0 = (kb - tap * cbt) * 64 + j * 8;
            ok = c0 < C;
        } else {
            const int q = kb * 8 + j;
            ok = q < nchunks;
            tap = ok ? q / cpt : 0;
            c0 = (q - tap * cpt) * 8;
        }
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (k < K && ok) {
            const int jk = k / Ko, jc = c0 / Co;        // original group within the super-group
            if (jk == jc) {
                const long long go = (long long)g * pack + jk;
                v = w[(((go * Ko + (k - jk * Ko)) * taps + tap) * Co + (c0 - jc * Co)) / 8];
            }
        }
        const long long tile = (((long long)g * num_nt + nt) * nkb + kb) * BN + n;
        out[tile * 8 + (j ^ (n & 7))] = v;
    }
}

// 3xTF32 layout: per (group, N tile, K block) a BN x 128-byte tile of the high parts
// (w with its low 13 mantissa bits cleared: exact in TF32) followed by the same tile of the
// low parts (w - high, exact in fp32), both 128-byte swizzled.  K block kb = tap*cbt + b
// holds channels 32b..32b+31 of that tap; 16-byte chunk j holds channels 32b+4j..+3.
__global__ void prepack_tf32x3_kernel(const float4* __restrict__ w, uint4* __restrict__ out, int K, int C,
                                      int taps, int BN, int num_nt, int nkb, int cbt, int slab_order, int Y, int X,
                                      long long total16) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total16;
         idx += (long long)gridDim.x * blockDim.x) {
        const int j = (int)(idx & 7);
        long long r = idx >> 3;
        const int n = (int)(r % BN); r /= BN;
        const int kb = (int)(r % nkb); r /= nkb;
        const int nt = (int)(r % num_nt);
        const int g = (int)(r / num_nt);
        const int k = nt * BN + n;
        int tap, c0;
        if (slab_order) {   // K block kb = ((z*cbt + b)*Y + y)*X + x, as for bf16
            const int kg = kb / (Y * X), t = kb - kg * (Y * X);
            const int z = kg / cbt, b = kg - z * cbt;
            tap = (z * Y + t / X) * X + t % X;
            c0 = b * 32 + j * 4;
        } else {
            tap = kb / cbt;
            c0 = (kb - tap * cbt) * 32 + j * 4;
        }
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < K && c0 < C) v = w[((((long long)g * K + k) * taps + tap) * C + c0) / 4];
        uint4 hi, lo;
        hi.x = __float_as_uint(v.x) & 0xFFFFE000u; hi.y = __float_as_uint(v.y) & 0xFFFFE000u;
        hi.z = __float_as_uint(v.z) & 0xFFFFE000u; hi.w = __float_as_uint(v.w) & 0xFFFFE000u;
        lo.x = __float_as_uint(v.x - __uint_as_float(hi.x)); lo.y = __float_as_uint(v.y - __uint_as_float(hi.y));
        lo.z = __float_as_uint(v.z - __uint_as_float(hi.z)); lo.w = __float_as_uint(v.w - __uint_as_float(hi.w));
        const long long tile = (((long long)g * num_nt + nt) * nkb + kb);
        const long long rowpos = (long long)n * 8 + (j ^ (n & 7));
        out[tile * 2 * BN * 8 + rowpos] = hi;
        out[tile * 2 * BN * 8 + (long long)BN * 8 + rowpos] = lo;
    }
}

// FFMA layout: [G][taps*C][Kpad], output channels contiguous, zero beyond K.
template <typename T>
__global__ void prepack_simt_kernel(const T* __restrict__ w, T* __restrict__ out, int K, int C, int taps, int Kg,
                                    int Kpad, long long total) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int n = (int)(idx % Kpad);
        const long long r = idx / Kpad;
        const int kk = (int)(r % Kg);
        const int g = (int)(r / Kg);
        const int tap = kk / C;
        const int c = kk - tap * C;
        out[idx] = n < K ? w[(((long long)g * K + n) * taps + tap) * C + c] : T(0.0f);
    }
}

// Backward data at unit stride: the forward weight of the transposed problem,
// w'[g][c][tap'][k] = w[g][k][taps-1-tap'][c] (every tap axis flipped, C and K swapped),
// element type E (2 or 4 bytes), staged for the forward prepack.
// For a stride phase the staged taps are a subset: staged tap t' = (z', y', x') of a Zs x Ys x Xs
// filter is forward tap (t0 - t'*dt) per axis of the Zo x Yo x Xo one.
struct TapMap {
    int Zo, Yo, Xo, Zs, Ys, Xs;
    int t0[3], dt[3];
};

template <typename E>
__global__ void flip_transpose_kernel(const E* __restrict__ w, E* __restrict__ out, int K, int C, TapMap tm,
                                      long long total) {
    const int taps_s = tm.Zs * tm.Ys * tm.Xs, taps_o = tm.Zo * tm.Yo * tm.Xo;
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int k = (int)(idx % K);
        long long r = idx / K;
        const int t = (int)(r % taps_s); r /= taps_s;
        const int c = (int)(r % C);
        const long long g = r / C;
        const int xs = t % tm.Xs, ys = (t / tm.Xs) % tm.Ys, zs = t / (tm.Xs * tm.Ys);
        const int tap = ((tm.t0[0] - zs * tm.dt[0]) * tm.Yo + (tm.t0[1] - ys * tm.dt[1])) * tm.Xo +
                        (tm.t0[2] - xs * tm.dt[2]);
        out[idx] = w[((g * K + k) * taps_o + tap) * C + c];
    }
}

// Backward data on the FFMA pipe: [G][taps*K][Cpad] with B[(tap, k)][c] = w[g][k][tap][c].
template <typename T>
__global__ void prepack_dg_simt_kernel(const T* __restrict__ w, T* __restrict__ out, int K, int C, int taps, int Kg,
                                       int Cpad, long long total) {
    for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * blockDim.x) {
        const int c = (int)(idx % Cpad);
        const long long r = idx / Cpad;
        const int kk = (int)(r % Kg);
        const int g = (int)(r / Kg);
        const int tap = kk / K;
        const int k = kk - tap * K;
        out[idx] = c < C ? w[(((long long)g * K + k) * taps + tap) * C + c] : T(0.0f);
    }
}

// fp32 -> three bf16 planes: hi = bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid).  Both
// differences are exact in fp32 (each has at most 16 significant bits), so hi + mid + lo equals
// v to within 2^-24 of it.  Plane p of element i at out[p * n + i].
__global__ void split_planes_kernel(const float* __restrict__ in, __nv_bfloat16* __restrict__ out, long long n) {
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
        const float v = __ldg(in + i);
        const __nv_bfloat16 h = __float2bfloat16_rn(v);
        const float r1 = v - __bfloat162float(h);
        const __nv_bfloat16 m = __float2bfloat16_rn(r1);
        const float r2 = r1 - __bfloat162float(m);
        out[i] = h;
        out[n + i] = m;
        out[2 * n + i] = __float2bfloat16_rn(r2);
    }
}

// ----------------------------------------------------------------------------- split-K reduction
// y = epilogue(sum over splits, in split order, of the fp32 partials): a fixed order,
// so results do not change from run to run.
__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ void from_f(float& d, float v) { d = v; }
__device__ __forceinline__ void from_f(__nv_bfloat16& d, float v) { d = __float2bfloat16_rn(v); }

// Row m of the partials (pixels in N Do Ho Wo order) -> its place in y.
__device__ __forceinline__ long long reduce_row(const Lattice& L, long long m, int Do, int Ho, int Wo) {
    if (!L.on) return m;
    const int ow = (int)(m % Wo);
    long long q = m / Wo;
    const int oh = (int)(q % Ho);
    q /= Ho;
    const int od = (int)(q % Do);
    return lattice_pixel(L, (int)(q / Do), od, oh, ow);
}

template <typename T>
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int splits, long long MGK, int GK,
                                     const T* __restrict__ bias, T* __restrict__ y, int epi, int pdl, Lattice lat,
                                     int Do, int Ho, int Wo) {
    if (pdl) {   // the partial sums come from the conv kernel just before this one
        griddep_launch();
        griddep_wait();
    }
    const bool add_bias = epi == EPI_BIAS || epi == EPI_BIAS_GELU;
    const bool do_gelu = epi == EPI_BIAS_GELU || epi == EPI_GELU;
    if ((GK & 3) == 0) {
        const long long n4 = MGK / 4;
        for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n4;
             i += (long long)gridDim.x * blockDim.x) {
            float4 a = __ldg(reinterpret_cast<const float4*>(ws) + i);
            for (int s = 1; s < splits; ++s) {
                const float4 b = __ldg(reinterpret_cast<const float4*>(ws + (long long)s * MGK) + i);
                a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
            }
            float v[4] = {a.x, a.y, a.z, a.w};
            const int col = (int)((i * 4) % GK);
            const long long o = reduce_row(lat, (i * 4) / GK, Do, Ho, Wo) * GK + col;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (add_bias) v[e] += to_f(bias[col + e]);
                if (do_gelu) v[e] = gelu(v[e]);
                from_f(y[o + e], v[e]);
            }
        }
    } else {
        for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < MGK;
             i += (long long)gridDim.x * blockDim.x) {
            float a = ws[i];
            for (int s = 1; s < splits; ++s) a += ws[(long long)s * MGK + i];
            if (add_bias) a += to_f(bias[i % GK]);
            if (do_gelu) a = gelu(a);
            from_f(y[reduce_row(lat, i / GK, Do, Ho, Wo) * GK + i % GK], a);
        }
    }
}

}  // namespace

// ----------------------------------------------------------------------------- plan
enum Variant { VAR_TC = 0, VAR_SIMT = 1, VAR_DG_SIMT = 2, VAR_WG_SIMT = 3, VAR_WG_TC = 4, VAR_DG_PHASED = 5 };
constexpr int MAX_PHASES = 16;
enum Direction { DIR_FWD = 0, DIR_BWD_DATA = 1, DIR_BWD_WEIGHT = 2 };

// Plan choices that can be fixed instead of decided by rule: by the measured selector
// (conv_plan_tune and its table) or, for tests, by CONV_FORCE_* environment variables.
// 0 (or -1 where 0 is a meaningful value) leaves the choice to the rules.
struct PlanChoice {
    int simt = 0;          // 1: the FFMA kernel
    int no_pack = 0;       // 1: never pack groups narrower than 64 channels
    int bn = 0;            // tensor-core N tile: 16, 32, 64, 128 or 256
    int bm = 0;            // FFMA M tile: 64 or 128
    int splits = 0;        // >= 1: split-K factor (capped by the K blocks)
    int gather = 0;        // 1: cp.async chunks (bf16), 2: per-tap TMA boxes (no slab)
    int slab_stream = 0;   // 1: slab mode streams its weights through a ring
    int slab_pair = -1;    // 0 / 1: slab tile pairs off / on
    int epi_warps = 0;     // 8 or 16 epilogue warps in the per-tap kernel
    int cluster_red = -1;  // 0: split-K partials through the reduction kernel, not a cluster
    int mc = -1;           // 0 / 1: CTA pairs sharing weight tiles by multicast off / on
    int pair = -1;         // 0 / 1: M = 256 tiles over CTA pairs (.cta_group::2 MMAs) off / on
    int ystore = -1;       // 0: per-lane stores of y even where a tensor-map (TMA) store could serve
    int slab_bw = 0;       // > 0: slab tiles this many output columns wide
    bool operator==(const PlanChoice& o) const {
        return simt == o.simt && no_pack == o.no_pack && bn == o.bn && bm == o.bm && splits == o.splits &&
               gather == o.gather && slab_stream == o.slab_stream && slab_pair == o.slab_pair &&
               epi_warps == o.epi_warps && cluster_red == o.cluster_red && mc == o.mc && pair == o.pair &&
               ystore == o.ystore && slab_bw == o.slab_bw;
    }
};

struct conv_plan {
    PlanChoice ch;
    int ndim;
    int64_t spatial[3], filter[3], stride[3], pad[3], dil[3], out_spatial[3];
    conv_dtype dtype;
    conv_epilogue epi;
    Geom g;
    int sm_count;
    Variant variant;
    // tensor-core plan
    int BN, stages, num_mt, num_nt, nkb, nchunks, cpt, splits, kbps, total_units, grid;
    int tma, map_kind, BW, BH, tiles_w, tiles_h, cbt, tf32, sleep_mask;
    int pack, Go, Co, Ko;   // small-group packing factor and the caller's G, C, K
    int slab, slab_bws, slab_hr, slab_nkg, slab_nbg, slab_btaps, slab_sa, slab_sb, slab_a_stage, slab_resident;
    int slab_nacc, slab_pair_rows, acc_bh;   // tile pairs (see set_slab_pair)
    int overlap;            // launch as programmatic dependents (conv_plan_set_overlap)
    int epi_warps;          // per-tap kernel epilogue warps (8 or 16)
    int cluster_red;        // split-K partials summed inside a cluster (no workspace, no reduce kernel)
    int mc;                 // CTA pairs share each weight tile by multicast (units are pairs of M tiles)
    int pair;               // M = 256 tiles over CTA pairs with .cta_group::2 MMAs (units are pairs of M tiles)
    int ystore;             // the epilogue stores y with TMA boxes (tiles of one output row)
    size_t slab_smem;
    // SIMT plan
    int BM, Kg, Kpad, nkt, ktps, vec;
    size_t prepack_bytes, workspace_bytes;
    size_t packed_bytes;    // the packed weight alone (prepack_bytes may add a staging area)
    void* workspace;
    size_t workspace_size;
    double flops;
    // backward plans
    int dir;                // Direction
    Geom fg;                // the forward problem (g is the problem the kernels run)
    int dg_fwd;             // backward data run as the forward conv of dy with flipped, transposed weights
    size_t dg_src_off;      // where in w_packed the prepack stages those weights
    int dg_t0[3], dg_dt[3]; // staged tap t' (per axis) is forward tap t0 - t'*dt
    Lattice lat;            // output placement (stride phases of a backward data)
    conv_plan* ph[MAX_PHASES];   // stride phases: forward plans whose outputs interleave in dx
    size_t ph_off[MAX_PHASES];   // each phase's packed weight within w_packed
    int nph;
    int ph_zero;            // some input pixels receive no tap at all: dx is cleared first
    int test_stall;         // CONV_TEST_STALL: the tensor-core kernel's MMA role waits until its bounded
                            // wait expires (exercises the timeout path; tests only)
    int wg_kt, wg_jt, wg_mps, wg_tile;   // backward weight (FFMA): tiles along K and taps*C, pixels per split, tile
    int wg_rt, wg_nt, wg_q, wg_qps, wg_nwb, wg_cbh, wg_pack;   // backward weight (tensor cores), see WgradTcParams
    int wg_planes;                      // 1 (bf16) or 3 (fp32 split into bf16 planes)
    int wg_slab, wg_na, wg_hpp, wg_nbox, wg_box_rows, wg_box_bytes, wg_stage_bytes, wg_stages, wg_tmem;   // slab mode
    size_t wg_xpl_off, wg_dypl_off;     // fp32: the x and dy planes within the workspace
    char desc[320];
};

static int env_int(const char* name, int dflt) {
    const char* v = getenv(name);
    if (!v || !*v) return dflt;
    return atoi(v);
}

// The test hooks: CONV_FORCE_* variables fix a choice; returns whether any was set.
static bool choice_from_env(PlanChoice& c) {
    bool any = false;
    auto take = [&](const char* name, int& field) {
        const char* v = getenv(name);
        if (v && *v) {
            field = atoi(v);
            any = true;
        }
    };
    take("CONV_FORCE_SIMT", c.simt);
    take("CONV_NO_PACK", c.no_pack);
    take("CONV_FORCE_BN", c.bn);
    take("CONV_FORCE_BM", c.bm);
    take("CONV_FORCE_SPLITK", c.splits);
    take("CONV_FORCE_SLAB_STREAM", c.slab_stream);
    take("CONV_FORCE_SLAB_PAIR", c.slab_pair);
    take("CONV_FORCE_EPI_WARPS", c.epi_warps);
    take("CONV_FORCE_CLUSTER_RED", c.cluster_red);
    take("CONV_FORCE_MC", c.mc);
    take("CONV_FORCE_PAIR", c.pair);
    take("CONV_FORCE_YSTORE", c.ystore);
    take("CONV_FORCE_SLAB_BW", c.slab_bw);
    if (const char* v = getenv("CONV_FORCE_GATHER")) {
        if (strcmp(v, "cpasync") == 0) { c.gather = 1; any = true; }
        else if (strcmp(v, "tma") == 0) { c.gather = 2; any = true; }
    }
    return any;
}

static int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

static int query_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return 152; }
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
        cudaGetLastError();
        return 152;
    }
    return n;
}

// ---- activation tensor map (TMA gather) ----
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static bool tried = false;
    static std::mutex mu;
    std::lock_guard<std::mutex> lk(mu);
    if (!tried) {
        tried = true;
        void* f = nullptr;
        void* init = nullptr;
        cudaDriverEntryPointQueryResult q;
        // the encoder needs an initialised driver, which a plan made before any CUDA
        // context exists would not have: initialise it (idempotent)
        if (cudaGetDriverEntryPointByVersion("cuInit", &init, 2000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess &&
            reinterpret_cast<PFN_cuInit_v2000>(init)(0) == CUDA_SUCCESS &&
            cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        else
            cudaGetLastError();
    }
    return fn;
}

// The input as a 5-D tensor for tiled TMA boxes of one 128-byte channel block (64 bf16 or
// 32 fp32 channels) x BW x BH output pixels:
// map_kind 0: {G*C, W, H, D, N} (C a multiple of the block, or G = 1: a box never reads another
// group's channels); map_kind 1: {C, G, W, H, N} (D = Z = 1).  The conv stride is the
// box's element stride; padding and the channel tail read as zero (out of range).
static bool encode_act_map(const conv_plan* p, const void* x, CUtensorMap* map) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const Geom& g = p->g;
    const cuuint64_t e = p->tf32 ? 4 : 2;         // fp32 or bf16
    const cuuint32_t cblk = p->tf32 ? 32 : 64;    // channels in one 128-byte row
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], es[5];
    // per-tap boxes cover BW x BH output pixels (stride as element stride); slab boxes cover
    // the tile's input rows: BWs x HR pixels at unit stride
    const cuuint32_t bx = p->slab ? (cuuint32_t)p->slab_bws : (cuuint32_t)(p->BW * g.sw);
    const cuuint32_t by = p->slab ? (cuuint32_t)p->slab_hr : (cuuint32_t)(p->BH * g.sh);
    const cuuint32_t ex = p->slab ? 1u : (cuuint32_t)g.sw, ey = p->slab ? 1u : (cuuint32_t)g.sh;
    if (p->map_kind == 0) {
        dims[0] = (cuuint64_t)g.G * g.C; dims[1] = g.W; dims[2] = g.H; dims[3] = g.D; dims[4] = g.N;
        strides[0] = dims[0] * e;
        strides[1] = strides[0] * g.W;
        strides[2] = strides[1] * g.H;
        strides[3] = strides[2] * g.D;
        box[0] = cblk; box[1] = bx; box[2] = by; box[3] = 1; box[4] = 1;
        es[0] = 1; es[1] = ex; es[2] = ey; es[3] = 1; es[4] = 1;
    } else {
        dims[0] = g.C; dims[1] = g.G; dims[2] = g.W; dims[3] = g.H; dims[4] = g.N;
        strides[0] = (cuuint64_t)g.C * e;
        strides[1] = (cuuint64_t)g.G * g.C * e;
        strides[2] = strides[1] * g.W;
        strides[3] = strides[2] * g.H;
        box[0] = cblk; box[1] = 1; box[2] = bx; box[3] = by; box[4] = 1;
        es[0] = 1; es[1] = 1; es[2] = ex; es[3] = ey; es[4] = 1;
    }
    const CUresult r = fn(map, p->tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5,
                          const_cast<void*>(x), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// The packed weights of a CTA-pair plan as a tensor of 128-byte rows (64 bf16) from which each
// CTA of a pair loads its half (BN/2 rows) of every weight tile: per-tap plans one tile per
// copy, slab plans all the tap tiles of a weight stage in one copy (a second copy from the same
// thread waits for the first, so one copy per tap made the first stages arrive microseconds
// late).  The rows are copied verbatim (they are already 128-byte swizzled by the prepack).
static bool encode_w_map(const conv_plan* p, const void* w_packed, CUtensorMap* map) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t tiles = (cuuint64_t)p->g.G * p->num_nt * p->nkb;
    const cuuint32_t half = (cuuint32_t)(p->BN / 2);
    CUresult r;
    if (p->slab) {
        // {64 channels, BN/2 rows, 2 halves, tap tiles}: a box of one half of `slab_btaps`
        // consecutive tap tiles is one slab weight stage of one CTA
        cuuint64_t dims[4] = {64, half, 2, tiles};
        cuuint64_t strides[3] = {128, (cuuint64_t)half * 128, (cuuint64_t)p->BN * 128};
        cuuint32_t box[4] = {64, half, 1, (cuuint32_t)p->slab_btaps};
        cuuint32_t es[4] = {1, 1, 1, 1};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(w_packed), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    } else {
        // {64 channels, rows}: a box of BN/2 rows is one CTA's half of a tap tile
        cuuint64_t dims[2] = {64, tiles * p->BN};
        cuuint64_t strides[1] = {128};
        cuuint32_t box[2] = {64, half};
        cuuint32_t es[2] = {1, 1};
        r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w_packed), dims, strides, box, es,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    }
    return r == CUDA_SUCCESS;
}

// y as a 5-D tensor {G*K, Wo, Ho, Do, N} for TMA stores of one warp's chunk, 64 or 32 channels
// x 32 pixels along Wo (bf16, 128- or 64-byte swizzle: the epilogue's staging layout).
static bool encode_y_map(const conv_plan* p, const void* y, CUtensorMap* map) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const Geom& g = p->g;
    cuuint64_t dims[5] = {(cuuint64_t)g.G * g.K, (cuuint64_t)g.Wo, (cuuint64_t)g.Ho, (cuuint64_t)g.Do, (cuuint64_t)g.N};
    cuuint64_t strides[4];
    strides[0] = dims[0] * 2;
    strides[1] = strides[0] * dims[1];
    strides[2] = strides[1] * dims[2];
    strides[3] = strides[2] * dims[3];
    const int cw = tc_store_cols(p->BN, p->epi_warps, p->pair != 0);
    cuuint32_t box[5] = {(cuuint32_t)cw, 32, 1, 1, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(y), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, cw == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Output tile BH x BW (<= 128 pixels of one output plane) that wastes the fewest MMA rows.
static void choose_tile_shape(conv_plan* p) {
    const Geom& g = p->g;
    int best_bw = 1, best_bh = 1;
    double best = -1.0;
    for (int k = 1; k <= 16; ++k) {
        const int bw = std::min<int64_t>(128, cdiv(g.Wo, k));
        if (bw * g.sw > 256) continue;
        int bh = std::max(1, std::min(g.Ho, 128 / bw));
        while (bh > 1 && bh * g.sh > 256) --bh;
        const double tiles = (double)cdiv(g.Wo, bw) * (double)cdiv(g.Ho, bh);
        const double eff = (double)g.Wo * g.Ho / (tiles * 128.0);
        if (eff > best + 1e-9) { best = eff; best_bw = bw; best_bh = bh; }
        if (bw == 1) break;
    }
    p->BW = best_bw;
    p->BH = best_bh;
    p->tiles_w = (int)cdiv(g.Wo, best_bw);
    p->tiles_h = (int)cdiv(g.Ho, best_bh);
}

// Slab geometry for a stride-1 problem (see tc_slab.cu): output tiles of BH rows x BW columns
// whose slab (BH + dh(Y-1)) x (BW + dw(X-1)) input pixels fit a 128-row accumulator.  Returns
// false when the problem has no such tile.
static bool set_slab_width(conv_plan* p, int bw);
static bool choose_slab_shape(conv_plan* p) {
    const Geom& g = p->g;
    const int reach_w = g.dw * (g.X - 1);
    int bw = std::min(g.Wo, 128 - reach_w);
    if (p->ch.slab_bw > 0) bw = std::min(bw, p->ch.slab_bw);
    if (bw < 8) return false;
    return set_slab_width(p, bw);
}

// Slab geometry for tiles bw output columns wide: as many output rows as fit a 128-row
// accumulator at the slab's row pitch bw + dw(X-1).
static bool set_slab_width(conv_plan* p, int bw) {
    const Geom& g = p->g;
    const int reach_w = g.dw * (g.X - 1), reach_h = g.dh * (g.Y - 1);
    const int bws = bw + reach_w;
    const int bh = std::max(1, std::min(g.Ho, 128 / bws));
    const int hr = bh + reach_h;
    if (bws > 256 || hr > 256) return false;
    p->BW = bw; p->BH = bh; p->acc_bh = bh; p->slab_nacc = 1; p->slab_pair_rows = 0;
    p->tiles_w = (int)cdiv(g.Wo, bw);
    p->tiles_h = (int)cdiv(g.Ho, bh);
    p->slab_bws = bws; p->slab_hr = hr;
    p->slab_nbg = g.Y; p->slab_btaps = g.X;
    // a window may read up to reach_h*bws + reach_w + 128 rows from the stage start
    const int64_t rows = std::max<int64_t>((int64_t)reach_h * bws + reach_w + 128, (int64_t)hr * bws);
    p->slab_a_stage = (int)(cdiv(rows * 128, 1024) * 1024 * (p->tf32 ? 2 : 1));
    return true;
}

// Slab geometry with one accumulator per unit (pair = false) or two stacked along H (pair =
// true): the unit covers 2 x acc_bh output rows and its slab the rows of both plus the filter's
// reach.  Returns false where the pair's box would exceed the 256-row TMA box limit.
static bool set_slab_pair(conv_plan* p, bool pair) {
    const Geom& g = p->g;
    const int reach_w = g.dw * (g.X - 1), reach_h = g.dh * (g.Y - 1);
    const int n = pair ? 2 : 1;
    const int hr = n * p->acc_bh + reach_h;
    if (hr > 256) return false;
    p->slab_nacc = n;
    p->BH = n * p->acc_bh;
    p->tiles_h = (int)cdiv(g.Ho, p->BH);
    p->slab_hr = hr;
    p->slab_pair_rows = pair ? p->acc_bh * p->slab_bws : 0;
    // the last window of the last accumulator starts at pair_rows + reach_h*bws + reach_w and
    // reads 128 rows
    const int64_t rows = std::max<int64_t>((int64_t)p->slab_pair_rows + (int64_t)reach_h * p->slab_bws + reach_w + 128,
                                           (int64_t)hr * p->slab_bws);
    p->slab_a_stage = (int)(cdiv(rows * 128, 1024) * 1024 * (p->tf32 ? 2 : 1));
    p->num_mt = g.N * g.Do * p->tiles_h * p->tiles_w;
    return true;
}

// Tensor-core tile choice: BN from the compiled set, the smallest padded width for K
// <= 256, else 256 or 128, whichever wastes fewer columns; then split-K when the tiles
// alone leave SMs idle (page "onnxruntime PR #33639", "Description": large tiles for
// large problems, split-K for small problems because it fills the GPU better).
static bool plan_tc(conv_plan* p, bool tf32, bool allow_slab = true);
static bool plan_tc_per_tap_retry(conv_plan* p, bool tf32) { return plan_tc(p, tf32, false); }

static bool plan_tc(conv_plan* p, bool tf32, bool allow_slab) {
    const Geom& g = p->g;
    int bn;
    if (g.K <= 16) bn = 16;
    else if (g.K <= 32) bn = 32;
    else if (g.K <= 64) bn = 64;
    else if (g.K <= 128) bn = 128;
    else if (g.K <= 256) bn = 256;
    else bn = (cdiv(g.K, 256) * 256 - g.K <= cdiv(g.K, 128) * 128 - g.K) ? 256 : 128;
    const int force_bn = p->ch.bn;
    if (force_bn == 16 || force_bn == 32 || force_bn == 64 || force_bn == 128 || force_bn == 256) bn = force_bn;
    p->tf32 = tf32 ? 1 : 0;
    p->BN = bn;
    p->epi_warps = 8;
    p->stages = tc_stages_for(bn, p->tf32, 8);
    p->cpt = g.C / 8;
    p->nchunks = g.taps * p->cpt;
    // Gather: TMA boxes when the tensor map can express the problem and a tap has at
    // least one full 128-byte channel block; otherwise (bf16 only) 16-byte cp.async chunks
    // packed densely across taps.
    const int cblk = tf32 ? 32 : 64;
    int map_kind = -1;
    if (g.C % cblk == 0 || g.G == 1) map_kind = 0;
    else if (g.D == 1 && g.Z == 1) map_kind = 1;
    bool tma = map_kind >= 0 && g.C >= cblk && g.sw <= 8 && g.sh <= 8;
    if (!tf32 && p->ch.gather == 1) tma = false;
    // Slab mode for stride-1 problems with several taps per plane (one box serves them all);
    // its shared-memory fit is checked once the N tile is known.
    p->slab = 0;
    const bool want_slab = allow_slab && !p->lat.on && tma && g.sw == 1 && g.sh == 1 && g.sd == 1 && g.Y * g.X >= 3 &&
                           p->ch.gather != 2;
    if (tma) {
        p->map_kind = map_kind;
        if (want_slab && choose_slab_shape(p)) p->slab = 1;
        else choose_tile_shape(p);
        // A trial encode with a placeholder address checks the box against the driver's
        // limits.  The encoder needs a current context: make the current device's primary
        // context current first (without a device the rules above decide alone).
        int dev = 0;
        if (encode_fn() && cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess) {
            CUtensorMap probe;
            if (!encode_act_map(p, reinterpret_cast<const void*>((uintptr_t)4096), &probe)) {
                if (p->slab) {
                    p->slab = 0;
                    choose_tile_shape(p);
                    if (!encode_act_map(p, reinterpret_cast<const void*>((uintptr_t)4096), &probe)) tma = false;
                } else {
                    tma = false;
                }
            }
        }
        cudaGetLastError();
    }
    if (tf32 && !tma) return false;   // 3xTF32 needs the TMA gather
    // the epilogue warps wait a whole main loop per tile: they sleep; the rest poll
    p->sleep_mask = env_int("CONV_WAIT_SLEEP", 2);
    p->tma = tma ? 1 : 0;
    if (tma) {
        p->cbt = (int)cdiv(g.C, cblk);
        p->nkb = g.taps * p->cbt;
        p->num_mt = g.N * g.Do * p->tiles_h * p->tiles_w;
    } else {
        p->map_kind = 0; p->BW = 128; p->BH = 1; p->tiles_w = p->tiles_h = 1; p->cbt = 0;
        p->nkb = (int)cdiv(p->nchunks, 8);
        p->num_mt = (int)cdiv(g.M, 128);
    }
    // Small problems: narrower N tiles first (more CTAs, one launch, no partial sums), unless
    // each tile would then run a long reduction (K blocks weighted by the MMAs per block: 3
    // for 3xTF32), where splitting K finishes sooner; split-K also when even 32-wide tiles
    // leave more than half the SMs idle.
    if (force_bn == 0 && p->nkb * (tf32 ? 3 : 1) <= 32) {
        while (bn > 32 && (int64_t)p->num_mt * g.G * cdiv(g.K, bn) * 4 < (int64_t)p->sm_count * 3) bn /= 2;
        p->BN = bn;
        p->stages = tc_stages_for(bn, p->tf32, 8);
    }
    p->num_nt = (int)cdiv(g.K, bn);
    int64_t units = (int64_t)p->num_mt * g.G * p->num_nt;
    int splits = 1;
    if (units * 2 < p->sm_count && p->nkb >= 4) {
        splits = (int)std::min<int64_t>(p->sm_count / units, p->nkb / 2);
        splits = std::max(1, std::min(splits, 16));
    }
    if (p->ch.splits >= 1) splits = std::min(p->ch.splits, p->nkb);
    if (p->slab) {
        // slab mode runs whole reductions per tile and needs its rings to fit: the weights of
        // one (group, N tile) resident with a 3- or 2-stage slab ring where they fit, else a
        // ring of weight stages
        p->slab_nkg = g.Z * p->cbt;
        const int nchunk = p->slab_nkg * p->slab_nbg;
        auto fit_rings = [&]() {
            p->slab_sa = 2;
            p->slab_sb = 0;
            p->slab_resident = 0;
            for (int sa = 3; sa >= 2 && !p->slab_resident; --sa)
                if (p->ch.slab_stream == 0 &&
                    slab_smem_bytes(bn, p->tf32, sa, nchunk, (size_t)p->slab_a_stage, p->slab_btaps) <= SLAB_SMEM_MAX) {
                    p->slab_resident = 1;
                    p->slab_sa = sa;
                    p->slab_sb = nchunk;
                }
            for (int sb = 8; sb >= 2 && !p->slab_resident; --sb)
                if (slab_smem_bytes(bn, p->tf32, 2, sb, (size_t)p->slab_a_stage, p->slab_btaps) <= SLAB_SMEM_MAX) {
                    p->slab_sb = sb;
                    break;
                }
            return p->slab_resident || p->slab_sb >= 2;
        };
        // Tile pairs (bf16, N tile <= 64, several units per CTA, more than one row block):
        // two accumulators per unit, stacked along H, share one slab and one weight pass.
        set_slab_pair(p, false);
        const int force_pair = p->ch.slab_pair;
        const bool want_pair = !tf32 && bn <= 64 && splits == 1 && g.Ho > p->acc_bh &&
                               (force_pair >= 0 ? force_pair == 1 : units >= 4LL * p->sm_count);
        bool fits = false;
        if (want_pair && set_slab_pair(p, true)) {
            fits = fit_rings();
            if (!fits) set_slab_pair(p, false);
        }
        if (!fits) fits = fit_rings();
        units = (int64_t)p->num_mt * g.G * p->num_nt;
        if (splits > 1 || !fits) {
            p->slab = 0;                               // back to per-tap boxes
            choose_tile_shape(p);
            return plan_tc_per_tap_retry(p, tf32);
        }
        p->slab_smem = slab_smem_bytes(bn, p->tf32, p->slab_sa, p->slab_sb, (size_t)p->slab_a_stage, p->slab_btaps);
    }
    p->kbps = (int)cdiv(p->nkb, splits);
    p->splits = (int)cdiv(p->nkb, p->kbps);     // every split non-empty
    // Wide bf16 tiles with short reductions (few K blocks per tile, e.g. 128 -> 1280 channels
    // at 3 taps) spend longer in the epilogue (bias, GELU, stores of BM x BN outputs) than in
    // the MMAs: they get 16 epilogue warps (4 per TMEM lane quarter), one stage fewer.
    if (!tf32 && p->tma && !p->slab && bn >= 128) {
        const int force_ew = p->ch.epi_warps;
        const bool wide_epi = force_ew ? force_ew == 16 : p->kbps <= 16;
        if (wide_epi) {
            p->epi_warps = 16;
            p->stages = tc_stages_for(bn, p->tf32, 16);
        }
    }
    p->total_units = (int)(units * p->splits);
    p->grid = std::min(p->total_units, p->sm_count);
    p->prepack_bytes = (size_t)g.G * p->num_nt * p->nkb * bn * 128 * (tf32 ? 2 : 1);
    // Split-K plans whose units all run at once (one per CTA) sum their partials inside a
    // thread-block cluster through distributed shared memory: no workspace, no second kernel.
    p->cluster_red = 0;
    if (p->splits >= 2 && p->splits <= 8 && (128 % p->splits) == 0 && p->total_units <= p->sm_count &&
        g.K % 4 == 0 && p->ch.cluster_red != 0)
        p->cluster_red = 1;
    p->workspace_bytes = (p->splits > 1 && !p->cluster_red) ? (size_t)p->splits * g.M * g.G * g.K * sizeof(float) : 0;
    // Weight multicast (bf16 per-tap TMA plans, N tiles of 128 or 256, no split): CTA pairs
    // compute M tiles 2j and 2j+1 of the same (group, N tile) together and read each weight
    // tile from L2 once per pair.  Only on request (the measured selector or CONV_FORCE_MC):
    // measured on the 128 -> 1280 -> 1280 conv1d layers at batch 32 the pairs' lockstep costs
    // more than the halved weight reads save (L1 105 -> 114 us, L2 309 -> 320 us).
    // CTA pairs with M = 256 MMAs (tc_pair.cu): bf16 per-tap TMA plans with N tiles of 128 or
    // 256, no split and long reductions (8 epilogue warps), when the pairs' units fill every
    // pair of SMs at least once.  Each SM then stores and reads half of every weight tile
    // (~64 KB instead of ~96 KB of shared-memory traffic per K block of 128x256 outputs).
    // Measured on the 128 -> 1280 -> 1280 conv1d at batch 32: the 60-block layer 309 -> 287 us;
    // the 6-block layer with 16 epilogue warps 102 -> 107 us, so plans with the wide epilogue
    // keep single CTAs unless forced.
    p->pair = 0;
    // Slab plans on CTA pairs (tc_slab_pair.cu): each CTA keeps its own slab and half of every
    // weight tile, and each M = 256 MMA reads a weight half per SM.  The rings are refitted for
    // half-size weight stages (resident weight sets where they fit, with a third slab stage
    // where possible).
    if (p->slab && !tf32 && (bn == 32 || bn == 64) && p->splits == 1 && !p->lat.on && p->ch.pair != 0) {
        const int nchunk = p->slab_nkg * p->slab_nbg;
        // three slab stages first (resident weights, else a ring of weight stages of one filter
        // row each), then two.  (Stages of one tap each, which would let more of them fit, were
        // measured 2.35x slower on the 3D d1 layer: four MMAs a stage cannot cover the pair's
        // hand-off of a stage.)
        int sa = 0, sb = 0, resident = 0;
        auto fit_pair_rings = [&]() {
            sa = sb = resident = 0;
            for (int a = 3; a >= 2 && !sa; --a) {
                if (p->ch.slab_stream == 0 &&
                    slab_pair_smem_bytes(bn, a, nchunk, (size_t)p->slab_a_stage, p->slab_btaps) <= SLAB_SMEM_MAX) {
                    sa = a; sb = nchunk; resident = 1;
                }
                for (int b = 8; b >= 2 && !sa; --b)
                    if (slab_pair_smem_bytes(bn, a, b, (size_t)p->slab_a_stage, p->slab_btaps) <= SLAB_SMEM_MAX) {
                        sa = a; sb = b;
                    }
            }
        };
        fit_pair_rings();
        // By rule pairs need three slab stages and a ring of at least four weight stages: a stage
        // is refilled only after both CTAs' copies of it were read, which shorter rings do not
        // cover, and with resident weights the units' epilogues (both CTAs') set the pace.
        // Measured (us per call, single CTA -> pair): 3D d1, 3 + 5 stages: 190.9 -> 137.4; 3D d2,
        // 3 + 2: 168.3 -> 331.7; 2D d2, 3 + 2: 39.9 -> 72.6; 2D d1, resident weights: 39.3 -> 39.8,
        // streamed (3 + 5): 39.3 -> 41.9.
        // Slab units of one accumulator per CTA run as pairs only on request (CONV_FORCE_PAIR=1
        // with a one-accumulator plan): each slab then serves half the MMAs, and on the 3D layers
        // they measured slower than single CTAs with tile pairs (d2, 3 + 5 stages: 164.2 ->
        // 182.4 us; d1: 137 -> 226 us against tile pairs).
        auto by_rule = [&]() { return p->num_mt >= 2 && sa >= 3 && !resident && sb >= 4 && p->slab_nacc == 2; };
        bool ok = by_rule() || (p->num_mt >= 2 && sa && p->ch.pair == 1);
        // A tile-pair slab too tall for that ring (dilation 2 in 3D: 8 input rows of 58 pixels
        // leave room for two weight stages) is made narrower instead: tiles of half the output
        // width hold twice the output rows, so the pair's slab has 12 rows of 31 pixels (47 KB
        // against 59 KB) and the ring of the dilation-1 layer fits.
        const int reach_w = g.dw * (g.X - 1);
        const conv_plan saved = *p;    // the single-CTA plan, restored if the pairs are not taken
        bool narrowed = false;
        if (!ok && !resident && p->slab_nacc == 2 && p->ch.pair != 1 && p->ch.slab_bw <= 0) {
            for (int k = 2; k <= 4 && !ok; ++k) {
                const int bw = (int)cdiv(g.Wo, k);
                if (bw < 8 || bw + reach_w > 128 || !set_slab_width(p, bw) || !set_slab_pair(p, true)) break;
                narrowed = true;
                fit_pair_rings();
                ok = by_rule();
            }
        }
        if (ok) {
            const int64_t pair_units = cdiv(p->num_mt, 2) * g.G * p->num_nt;
            const size_t smem = slab_pair_smem_bytes(bn, sa, sb, (size_t)p->slab_a_stage, p->slab_btaps);
            int clusters = p->sm_count / 2;
            int dev = 0;
            if (cudaGetDevice(&dev) == cudaSuccess) {
                const int n = slab_pair_max_clusters(smem);
                if (n > 0) clusters = std::min(clusters, n);
            }
            cudaGetLastError();
            // resident weights stay loaded only if a cluster keeps its (group, N tile): pair
            // units advance by the cluster count, so make it a multiple of the number of sets
            const int KT = g.G * p->num_nt;
            if (resident && KT <= clusters) clusters -= clusters % KT;
            if (clusters >= 1 && (p->ch.pair == 1 || pair_units >= clusters)) {
                p->pair = 1;
                p->slab_sa = sa; p->slab_sb = sb; p->slab_resident = resident;
                p->slab_smem = smem;
                p->total_units = (int)pair_units;
                p->grid = 2 * (int)std::min<int64_t>(pair_units, clusters);
                p->prepack_bytes = (size_t)g.G * p->num_nt * p->nkb * bn * 128;
            }
        }
        if (narrowed && !p->pair) *p = saved;   // the narrow tiles were only for the pairs
    }
    if (!tf32 && p->tma && !p->slab && p->splits == 1 && !p->cluster_red && (bn == 128 || bn == 256) &&
        p->num_mt >= 2 && p->ch.mc != 1) {
        const int64_t pair_units = cdiv(p->num_mt, 2) * g.G * p->num_nt;
        int clusters = p->sm_count / 2;
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) {
            const int n = tc_pair_max_clusters(bn, p->epi_warps);
            if (n > 0) clusters = std::min(clusters, n);
        }
        cudaGetLastError();
        if (clusters >= 1 && (p->ch.pair >= 0 ? p->ch.pair == 1 : (p->epi_warps == 8 && pair_units >= clusters))) {
            p->pair = 1;
            p->stages = tc_pair_stages_for(bn, p->epi_warps);
            p->total_units = (int)pair_units;
            p->grid = 2 * (int)std::min<int64_t>(pair_units, clusters);
        }
    }
    p->mc = 0;
    if (!tf32 && p->tma && !p->slab && p->splits == 1 && !p->cluster_red && bn >= 128 && p->num_mt >= 2 &&
        !p->pair && p->ch.mc == 1) {
        int clusters = p->sm_count / 2;
        int dev = 0;
        if (cudaGetDevice(&dev) == cudaSuccess) {
            const int n = tc_mc_max_clusters(bn, p->epi_warps);
            if (n > 0) clusters = std::min(clusters, n);
        }
        cudaGetLastError();
        if (clusters >= 1) {
            p->mc = 1;
            p->total_units = (int)(cdiv(p->num_mt, 2) * g.G * p->num_nt);
            p->grid = 2 * std::min(p->total_units, clusters);
        }
    }
    // Epilogue stores through a tensor map of y (bf16 per-tap plans, no split, tiles of one output
    // row whose width is a multiple of 32, chunks of 64 or 32 columns per warp, and columns that
    // never run into the next group): each warp's staged 32-row block leaves as one TMA store.  By
    // rule where CTAs run several tiles (measured on the conv1d sweep: 128 -> 1280 at batch 32
    // 107.0 -> 102.2 us; at batch 1, one tile per CTA, the final wait for the stores made it
    // 0.6 us slower).
    p->ystore = 0;
    if (!tf32 && p->tma && !p->slab && p->splits == 1 && !p->cluster_red && !p->lat.on && p->BH == 1 &&
        p->BW % 32 == 0 && (g.G == 1 || g.K % 64 == 0) && tc_store_cols(bn, p->epi_warps, p->pair != 0) >= 32 &&
        (p->ch.ystore >= 0 ? p->ch.ystore == 1 : p->total_units > p->sm_count))
        p->ystore = 1;
    if (p->slab)
        snprintf(p->desc, sizeof(p->desc),
                 "variant=%s gather=tma-slab tile=%dx%d pixels=%dx%d slab=%dx%d k_block=%d stages=%d+%d%s splits=1 "
                 "units=%d grid=%d k_blocks=%d map=%d acc=%d",
                 tf32 ? "tc_tf32x3" : "tc_bf16", 128 * p->slab_nacc, bn, p->BH, p->BW, p->slab_hr, p->slab_bws, cblk,
                 p->slab_sa, p->slab_resident ? 1 : p->slab_sb, p->slab_resident ? "w" : "", p->total_units, p->grid,
                 p->nkb, p->map_kind, p->slab_nacc);
    else if (p->tma)
        snprintf(p->desc, sizeof(p->desc),
                 "variant=%s gather=tma tile=128x%d pixels=%dx%d k_block=%d stages=%d splits=%d units=%d "
                 "grid=%d k_blocks=%d map=%d epi_warps=%d reduce=%s%s",
                 tf32 ? "tc_tf32x3" : "tc_bf16", bn, p->BH, p->BW, cblk, p->stages, p->splits, p->total_units,
                 p->grid, p->nkb, p->map_kind, p->epi_warps,
                 p->splits == 1 ? "none" : p->cluster_red ? "cluster" : "kernel",
                 p->pair ? " cta_pair=m256" : p->mc ? " weights=multicast2" : "");
    else
        snprintf(p->desc, sizeof(p->desc),
                 "variant=tc_bf16 gather=cp.async tile=128x%d k_block=64 stages=%d splits=%d units=%d grid=%d "
                 "k_blocks=%d",
                 bn, p->stages, p->splits, p->total_units, p->grid, p->nkb);
    if (p->slab && p->pair) {
        const size_t n = strlen(p->desc);
        snprintf(p->desc + n, sizeof(p->desc) - n, " cta_pair=m256");
    }
    if (p->ystore) {
        const size_t n = strlen(p->desc);
        snprintf(p->desc + n, sizeof(p->desc) - n, " store=tma");
    }
    return true;
}

static void plan_simt(conv_plan* p) {
    const Geom& g = p->g;
    p->Kg = g.taps * g.C;
    p->nkt = (int)cdiv(p->Kg, 8);
    p->num_nt = (int)cdiv(g.K, 128);
    p->Kpad = p->num_nt * 128;
    const int64_t tiles128 = cdiv(g.M, 128) * p->num_nt * g.G;
    p->BM = tiles128 >= p->sm_count ? 128 : 64;
    if (p->ch.bm == 64 || p->ch.bm == 128) p->BM = p->ch.bm;
    p->num_mt = (int)cdiv(g.M, p->BM);
    const int64_t tiles = (int64_t)p->num_mt * p->num_nt * g.G;
    int splits = 1;
    if (tiles < p->sm_count && p->nkt >= 32) {
        splits = (int)std::min<int64_t>(p->sm_count / tiles, p->nkt / 16);
        splits = std::max(1, std::min(splits, 16));
    }
    if (p->ch.splits >= 1) splits = std::min(p->ch.splits, p->nkt);
    p->ktps = (int)cdiv(p->nkt, splits);
    p->splits = (int)cdiv(p->nkt, p->ktps);
    p->vec = (g.C % 4 == 0 && g.K % 4 == 0) ? 1 : 0;
    const size_t esz = p->dtype == CONV_BF16 ? 2 : 4;
    p->prepack_bytes = (size_t)g.G * p->Kg * p->Kpad * esz;
    p->workspace_bytes = p->splits > 1 ? (size_t)p->splits * g.M * g.G * g.K * sizeof(float) : 0;
    snprintf(p->desc, sizeof(p->desc),
             "variant=simt_%s tile=%dx128 k_step=8 splits=%d grid=%dx%dx%d vec=%d",
             p->dtype == CONV_BF16 ? "bf16" : "f32", p->BM, p->splits, p->num_mt, p->num_nt,
             g.G * p->splits, p->vec);
}

static size_t align256(size_t n) { return (n + 255) & ~(size_t)255; }

// Variant and tiling of a plan whose geometry is set, under its choices p->ch (re-run by the
// selector with other choices).  Starts from the caller's geometry (Go, Co, Ko).
static void choose_variant(conv_plan* p) {
    Geom& g = p->g;
    const int64_t G = p->Go, C = p->Co, K = p->Ko;
    g.G = (int)G; g.C = (int)C; g.K = (int)K;
    p->pack = 1; p->slab = 0; p->tma = 0; p->cluster_red = 0; p->mc = 0; p->pair = 0; p->ystore = 0; p->epi_warps = 8;
    p->splits = 1;
    // bf16 with C, K multiples of 8: tcgen05 kind::f16.  fp32 with C, K multiples of 4 that the
    // TMA gather can express: tcgen05 3xTF32.  Everything else: the FFMA kernel.
    const bool no_tc = p->ch.simt != 0;
    bool tc = false;
    // Groups narrower than one 64-channel block: pack 64/C of them into a super-group with a
    // block-diagonal weight, so each tap still fills a whole 128-byte TMA box row (the MMA
    // does pack-fold redundant work on the zero blocks; the useful FLOP count is unchanged).
    if (!no_tc && p->dtype == CONV_BF16 && C % 8 == 0 && K % 8 == 0 && C < 64 && 64 % C == 0 &&
        G % (64 / C) == 0 && K * (64 / C) <= 4096 && p->ch.no_pack == 0) {
        p->pack = (int)(64 / C);
        g.G = (int)(G / p->pack); g.C = 64; g.K = (int)(K * p->pack);
    }
    if (!no_tc && p->dtype == CONV_BF16 && C % 8 == 0 && K % 8 == 0) tc = plan_tc(p, false);
    if (!tc && p->pack > 1) {   // not planned on the tensor cores after all: the caller's geometry
        p->pack = 1; g.G = (int)G; g.C = (int)C; g.K = (int)K;
    }
    if (!no_tc && p->dtype == CONV_F32 && C % 4 == 0 && K % 4 == 0) tc = plan_tc(p, true);
    if (tc) {
        p->variant = VAR_TC;
        if (p->pack > 1) {
            const size_t n = strlen(p->desc);
            snprintf(p->desc + n, sizeof(p->desc) - n, " pack=%d", p->pack);
        }
    } else {
        p->variant = VAR_SIMT;
        p->pack = 1; g.G = (int)G; g.C = (int)C; g.K = (int)K;
        plan_simt(p);
    }
    p->packed_bytes = p->prepack_bytes;
    if (p->dg_fwd) {   // the flipped, transposed weights are staged behind the packed ones
        p->dg_src_off = align256(p->prepack_bytes);
        p->prepack_bytes = p->dg_src_off + (size_t)G * C * K * p->g.taps * (p->dtype == CONV_BF16 ? 2 : 4);
        const size_t n = strlen(p->desc);
        snprintf(p->desc + n, sizeof(p->desc) - n, " direction=bwd_data(transposed_forward)");
    }
}

// ----------------------------------------------------------------------------- measured selector
// A process-wide table from a problem (its geometry, dtype, epilogue and the device's SM count)
// to the choices the selector measured fastest; conv_plan_create consults it.
static std::mutex g_tune_mu;
struct TuneEntry {
    PlanChoice c;
    double us = -1.0;                                    // measured time of the choice (-1: loaded)
    std::vector<std::pair<std::string, double>> log;     // every candidate timed: plan, us per call
};
static std::map<std::string, TuneEntry> g_tune_table;

static std::string plan_key(const conv_plan* p) {
    char buf[400];
    snprintf(buf, sizeof(buf),
             "nd=%d N=%d G=%lld C=%lld K=%lld in=%lldx%lldx%lld f=%lldx%lldx%lld s=%lldx%lldx%lld p=%lldx%lldx%lld "
             "d=%lldx%lldx%lld dtype=%d epi=%d dir=%d sm=%d",
             p->ndim, p->g.N, (long long)p->Go, (long long)p->Co, (long long)p->Ko, (long long)p->spatial[0],
             (long long)p->spatial[1], (long long)p->spatial[2], (long long)p->filter[0], (long long)p->filter[1],
             (long long)p->filter[2], (long long)p->stride[0], (long long)p->stride[1], (long long)p->stride[2],
             (long long)p->pad[0], (long long)p->pad[1], (long long)p->pad[2], (long long)p->dil[0],
             (long long)p->dil[1], (long long)p->dil[2], (int)p->dtype, (int)p->epi, p->dir, p->sm_count);
    return buf;
}

static void tune_table_lookup(const conv_plan* p, PlanChoice& c) {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    auto it = g_tune_table.find(plan_key(p));
    if (it != g_tune_table.end()) c = it->second.c;
}

// The candidates the selector times: the rules' own plan, each N tile x split factor x
// gather mode, CTA pairs and weight multicast for wide tiles, slab units of one or two
// accumulators on one CTA or a pair for narrow ones, and the FFMA kernel; candidates that land
// on the same plan are timed once.
static std::vector<conv_plan> tune_candidates(const conv_plan* p) {
    std::vector<PlanChoice> cs;
    cs.push_back(PlanChoice{});
    for (int bn : {32, 64, 128, 256})
        for (int sp : {1, 2, 4})
            for (int ga : {0, 2}) {
                PlanChoice c;
                c.bn = bn; c.splits = sp; c.gather = ga;
                cs.push_back(c);
            }
    for (int bn : {128, 256}) {    // wide unsplit tiles: one CTA, CTA pairs, or weight multicast
        PlanChoice c;
        c.bn = bn; c.splits = 1;
        c.pair = 0; cs.push_back(c);
        c.pair = 1; cs.push_back(c);
        c.pair = 0; c.mc = 1; cs.push_back(c);
    }
    for (int bn : {32, 64})        // slab units of one or two accumulators, on one CTA or a pair
        for (int tp : {0, 1})
            for (int pr : {0, 1}) {
                PlanChoice c;
                c.bn = bn; c.splits = 1; c.slab_pair = tp; c.pair = pr;
                cs.push_back(c);
            }
    PlanChoice f;
    f.simt = 1;
    cs.push_back(f);
    std::vector<conv_plan> out;
    for (const PlanChoice& c : cs) {
        conv_plan t = *p;
        t.ch = c;
        t.workspace = nullptr;
        t.workspace_size = 0;
        choose_variant(&t);
        bool seen = false;
        for (const conv_plan& o : out) seen = seen || strcmp(o.desc, t.desc) == 0;
        if (!seen) out.push_back(t);
    }
    return out;
}

// Validation and the forward geometry shared by the three plan kinds; on success *pp is a
// new plan with g = fg = the forward problem.
static conv_status init_plan(conv_plan** pp, conv_plan_t* out, int ndim, int64_t N, int64_t G, int64_t C, int64_t K,
                             const int64_t* spatial, const int64_t* filter, const int64_t* stride, const int64_t* pad,
                             const int64_t* dilation, conv_dtype dtype) {
    if (!out) return CONV_ERR_INVALID_ARG;
    if (ndim < 1 || ndim > 3 || !spatial || !filter || !stride || !pad || !dilation) return CONV_ERR_INVALID_ARG;
    if (N < 1 || G < 1 || C < 1 || K < 1) return CONV_ERR_INVALID_ARG;
    if (dtype != CONV_F32 && dtype != CONV_BF16) return CONV_ERR_INVALID_ARG;
    int64_t sp[3] = {1, 1, 1}, fl[3] = {1, 1, 1}, st[3] = {1, 1, 1}, pa[3] = {0, 0, 0}, di[3] = {1, 1, 1},
            os[3];
    const int off = 3 - ndim;   // conv1d -> D = H = 1, conv2d -> D = 1
    for (int i = 0; i < ndim; ++i) {
        if (spatial[i] < 1 || filter[i] < 1 || stride[i] < 1 || pad[i] < 0 || dilation[i] < 1)
            return CONV_ERR_INVALID_ARG;
        sp[off + i] = spatial[i]; fl[off + i] = filter[i]; st[off + i] = stride[i];
        pa[off + i] = pad[i]; di[off + i] = dilation[i];
    }
    const int64_t LIM = (int64_t)1 << 30;
    for (int i = 0; i < 3; ++i) {
        if (sp[i] > LIM || fl[i] > LIM || st[i] > LIM || pa[i] > LIM || di[i] > LIM) return CONV_ERR_UNSUPPORTED;
        const int64_t span = sp[i] + 2 * pa[i] - di[i] * (fl[i] - 1) - 1;
        if (span < 0) return CONV_ERR_INVALID_ARG;   // empty output
        os[i] = span / st[i] + 1;
    }
    if (N > LIM || G > LIM || C > LIM || K > LIM) return CONV_ERR_UNSUPPORTED;
    const int64_t M = N * os[0] * os[1] * os[2];
    const int64_t taps = fl[0] * fl[1] * fl[2];
    // the kernels index pixels, channels-by-taps and K blocks in 32 bits
    if (M >= ((int64_t)1 << 31) - 256 || taps * C >= ((int64_t)1 << 30) || G * C >= ((int64_t)1 << 30) ||
        G * K >= ((int64_t)1 << 30) || N * sp[0] * sp[1] * sp[2] >= ((int64_t)1 << 40))
        return CONV_ERR_UNSUPPORTED;

    conv_plan* p = new (std::nothrow) conv_plan();
    if (!p) return CONV_ERR_INVALID_ARG;
    p->ndim = ndim;
    for (int i = 0; i < 3; ++i) {
        p->spatial[i] = sp[i]; p->filter[i] = fl[i]; p->stride[i] = st[i];
        p->pad[i] = pa[i]; p->dil[i] = di[i]; p->out_spatial[i] = os[i];
    }
    p->dtype = dtype;
    Geom& g = p->g;
    g.N = (int)N; g.G = (int)G; g.C = (int)C; g.K = (int)K;
    g.D = (int)sp[0]; g.H = (int)sp[1]; g.W = (int)sp[2];
    g.Z = (int)fl[0]; g.Y = (int)fl[1]; g.X = (int)fl[2];
    g.sd = (int)st[0]; g.sh = (int)st[1]; g.sw = (int)st[2];
    g.pd = (int)pa[0]; g.ph = (int)pa[1]; g.pw = (int)pa[2];
    g.dd = (int)di[0]; g.dh = (int)di[1]; g.dw = (int)di[2];
    g.Do = (int)os[0]; g.Ho = (int)os[1]; g.Wo = (int)os[2];
    g.M = (int)M;
    g.taps = (int)taps;
    p->fg = g;
    // useful FLOPs of the forward problem; each backward pass does the same number
    p->flops = 2.0 * (double)M * (double)G * (double)K * (double)taps * (double)C;
    p->sm_count = query_sm_count();
    p->Go = g.G; p->Co = g.C; p->Ko = g.K;
    *pp = p;
    return CONV_OK;
}

static int gcd_int(int a, int b) { return b ? gcd_int(b, a % b) : a; }

// Backward data at stride > 1 as stride phases.  The input pixels i = r + s*j of one residue r
// (per axis) receive exactly the taps t with (r + pad - t*dil) divisible by s, from output
// position j + q_t, q_t = (r + pad - t*dil)/s.  Those taps are every (s / gcd(s, dil))-th one,
// so a phase is a unit-stride forward convolution of dy with the subset of taps reversed,
// dilation dil / gcd(s, dil) and padding -q of the last tap, C and K swapped, whose outputs land
// on the lattice r + s*j of dx.  Each phase runs the tensor-core forward kernels; a residue that
// no tap reaches leaves zeros (dx is cleared first).  Returns false where a phase does not fit
// the tensor-core path (the gather kernel is used instead).
static bool plan_dg_phased(conv_plan* p) {
    const Geom& f = p->fg;
    const int S[3] = {f.sd, f.sh, f.sw}, P[3] = {f.pd, f.ph, f.pw}, DL[3] = {f.dd, f.dh, f.dw};
    const int F[3] = {f.Z, f.Y, f.X}, I[3] = {f.D, f.H, f.W}, O[3] = {f.Do, f.Ho, f.Wo};
    if ((int64_t)S[0] * S[1] * S[2] > MAX_PHASES) return false;
    if (p->dtype == CONV_BF16 ? (f.C % 8 || f.K % 8) : (f.C % 4 || f.K % 4)) return false;
    // per axis and residue: taps, first (largest) tap, tap step, padding, dilation, lattice size
    struct Axis { int nt, t0, dt, pad, dil, J; };
    Axis ax[3][8];
    for (int a = 0; a < 3; ++a) {
        if (S[a] > 8) return false;
        const int gg = gcd_int(S[a], DL[a]);
        for (int r = 0; r < S[a]; ++r) {
            Axis& A = ax[a][r];
            A.J = r < I[a] ? (I[a] - r + S[a] - 1) / S[a] : 0;
            A.nt = 0; A.t0 = -1;
            for (int t = F[a] - 1; t >= 0; --t) {
                const int num = r + P[a] - t * DL[a];
                if (((num % S[a]) + S[a]) % S[a] == 0) {
                    if (A.t0 < 0) A.t0 = t;
                    ++A.nt;
                }
            }
            A.dt = S[a] / gg;
            A.dil = DL[a] / gg;
            A.pad = A.t0 >= 0 ? -((r + P[a] - A.t0 * DL[a]) / S[a]) : 0;
        }
    }
    p->nph = 0;
    p->ph_zero = 0;
    size_t off = 0, ws = 0;
    bool ok = true;
    for (int rd = 0; rd < S[0] && ok; ++rd)
        for (int rh = 0; rh < S[1] && ok; ++rh)
            for (int rw = 0; rw < S[2] && ok; ++rw) {
                const Axis* A[3] = {&ax[0][rd], &ax[1][rh], &ax[2][rw]};
                if (!A[0]->J || !A[1]->J || !A[2]->J) continue;             // no pixels in this residue
                if (!A[0]->nt || !A[1]->nt || !A[2]->nt) { p->ph_zero = 1; continue; }
                conv_plan* q = new (std::nothrow) conv_plan(*p);
                if (!q) { ok = false; break; }
                q->nph = 0;
                Geom& g = q->g;
                g.C = f.K; g.K = f.C;
                g.D = f.Do; g.H = f.Ho; g.W = f.Wo;
                g.Z = A[0]->nt; g.Y = A[1]->nt; g.X = A[2]->nt;
                g.sd = g.sh = g.sw = 1;
                g.pd = A[0]->pad; g.ph = A[1]->pad; g.pw = A[2]->pad;
                g.dd = A[0]->dil; g.dh = A[1]->dil; g.dw = A[2]->dil;
                g.Do = A[0]->J; g.Ho = A[1]->J; g.Wo = A[2]->J;
                g.M = f.N * g.Do * g.Ho * g.Wo;
                g.taps = g.Z * g.Y * g.X;
                q->Go = g.G; q->Co = g.C; q->Ko = g.K;
                q->dg_fwd = 1;
                for (int a = 0; a < 3; ++a) { q->dg_t0[a] = A[a]->t0; q->dg_dt[a] = A[a]->dt; }
                q->lat.on = 1;
                q->lat.D = f.D; q->lat.H = f.H; q->lat.W = f.W;
                q->lat.sd = S[0]; q->lat.sh = S[1]; q->lat.sw = S[2];
                q->lat.rd = rd; q->lat.rh = rh; q->lat.rw = rw;
                q->workspace = nullptr; q->workspace_size = 0;
                choose_variant(q);
                p->ph[p->nph++] = q;
                if (q->variant != VAR_TC) { ok = false; break; }
                p->ph_off[p->nph - 1] = off;
                off += align256(q->prepack_bytes);
                ws = std::max(ws, q->workspace_bytes);
            }
    if (!ok || p->nph == 0) {
        for (int i = 0; i < p->nph; ++i) delete p->ph[i];
        p->nph = 0;
        return false;
    }
    p->variant = VAR_DG_PHASED;
    p->prepack_bytes = p->packed_bytes = off;
    p->workspace_bytes = ws;
    const conv_plan* big = p->ph[0];
    for (int i = 1; i < p->nph; ++i)
        if (p->ph[i]->flops > big->flops) big = p->ph[i];
    // "variant=<the largest phase's> direction=bwd_data(phases) phases=P zero_fill=Z largest=<its other
    // fields, ':' for '=' and ',' for ' '>" (one key=value token each)
    const char* sp = strchr(big->desc, ' ');
    const int vlen = sp ? (int)(sp - big->desc) : (int)strlen(big->desc);
    int n = snprintf(p->desc, sizeof(p->desc), "%.*s direction=bwd_data(phases) phases=%d zero_fill=%d largest=", vlen,
                     big->desc, p->nph, p->ph_zero);
    for (const char* c = sp ? sp + 1 : ""; *c && n + 1 < (int)sizeof(p->desc); ++c) {
        if (strncmp(c, "direction=", 10) == 0) break;
        p->desc[n++] = *c == ' ' ? ',' : *c == '=' ? ':' : *c;
    }
    while (n > 0 && p->desc[n - 1] == ',') --n;
    p->desc[n] = 0;
    return true;
}

// Backward data on the FFMA pipe: rows are the N*D*H*W input pixels, columns the C input
// channels of a group, the reduction index tap*K + k; packed weight [G][taps*K][Cpad].
static void plan_dg_simt(conv_plan* p) {
    const Geom& f = p->fg;
    p->variant = VAR_DG_SIMT;
    const int rows = f.N * f.D * f.H * f.W;
    p->Kg = f.taps * f.K;
    p->nkt = (int)cdiv(p->Kg, 8);
    p->num_nt = (int)cdiv(f.C, 128);
    p->Kpad = p->num_nt * 128;
    const int64_t tiles128 = cdiv(rows, 128) * p->num_nt * f.G;
    p->BM = tiles128 >= p->sm_count ? 128 : 64;
    p->num_mt = (int)cdiv(rows, p->BM);
    const int64_t tiles = (int64_t)p->num_mt * p->num_nt * f.G;
    int splits = 1;
    if (tiles < p->sm_count && p->nkt >= 32) {
        splits = (int)std::min<int64_t>(p->sm_count / tiles, p->nkt / 16);
        splits = std::max(1, std::min(splits, 16));
    }
    p->ktps = (int)cdiv(p->nkt, splits);
    p->splits = (int)cdiv(p->nkt, p->ktps);
    p->vec = (f.C % 4 == 0 && f.K % 4 == 0) ? 1 : 0;
    const size_t esz = p->dtype == CONV_BF16 ? 2 : 4;
    p->prepack_bytes = (size_t)f.G * p->Kg * p->Kpad * esz;
    p->packed_bytes = p->prepack_bytes;
    p->workspace_bytes = p->splits > 1 ? (size_t)p->splits * rows * f.G * f.C * sizeof(float) : 0;
    snprintf(p->desc, sizeof(p->desc),
             "variant=simt_%s direction=bwd_data(gather) tile=%dx128 k_step=8 splits=%d grid=%dx%dx%d vec=%d",
             p->dtype == CONV_BF16 ? "bf16" : "f32", p->BM, p->splits, p->num_mt, p->num_nt, f.G * p->splits, p->vec);
}

// The two tensor maps of the tensor-core backward weight: x as {G*C, W, H, D, N} with boxes of
// 64 channels x 64 pixels at the conv stride along W, dy as {G*K, Wo, Ho, Do, N} with boxes of
// 64 channels x 64 output pixels; bf16, 128-byte swizzle, out-of-range elements read as zero.
static bool encode_wg_maps(const conv_plan* p, const void* x, const void* dy, CUtensorMap* xm, CUtensorMap* dym) {
    PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return false;
    const Geom& g = p->fg;
    cuuint64_t dims[5], strides[4];
    cuuint32_t box[5], es[5];
    const cuuint64_t images = (cuuint64_t)g.N * (p->wg_planes > 1 ? p->wg_planes : 1);   // plane pl, image n: pl*N + n
    dims[0] = (cuuint64_t)g.G * g.C; dims[1] = g.W; dims[2] = g.H; dims[3] = g.D; dims[4] = images;
    strides[0] = dims[0] * 2; strides[1] = strides[0] * g.W; strides[2] = strides[1] * g.H; strides[3] = strides[2] * g.D;
    box[0] = 64; box[1] = (cuuint32_t)(p->wg_slab ? p->wg_box_rows : 64 * g.sw); box[2] = box[3] = box[4] = 1;
    es[0] = 1; es[1] = (cuuint32_t)(p->wg_slab ? 1 : g.sw); es[2] = es[3] = es[4] = 1;
    if (fn(xm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(x), dims, strides, box, es,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return false;
    dims[0] = (cuuint64_t)g.G * g.K; dims[1] = g.Wo; dims[2] = g.Ho; dims[3] = g.Do; dims[4] = images;
    strides[0] = dims[0] * 2; strides[1] = strides[0] * g.Wo; strides[2] = strides[1] * g.Ho;
    strides[3] = strides[2] * g.Do;
    box[1] = 64;
    es[1] = 1;
    return fn(dym, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(dy), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Backward weight on the tensor cores (bf16, C and K multiples of 8 so that every box starts on a
// 16-byte boundary, stride along W at most 4 so a box spans <= 256 elements): 128-row tiles of (tap, 64-channel
// block) pairs x BN output channels; 64-pixel chunks along output rows split across CTAs until
// the grid fills the SMs once.  Returns false where the problem does not fit.
static bool plan_wg_tc(conv_plan* p) {
    const Geom& f = p->fg;
    if (p->ch.simt) return false;
    // fp32: x and dy split into three bf16 planes each (six plane products per tile)
    p->wg_planes = p->dtype == CONV_F32 ? 3 : 1;
    // every box starts at channel g*C + 64*b (x) or g*K + 64*j (dy): a multiple of 8 elements,
    // the 16-byte alignment a tiled TMA copy needs of its innermost coordinate
    if (f.C % 8 != 0 || f.K % 8 != 0 || f.sw > 4) return false;
    // groups narrower than half a box: `pack` groups share each box (block-diagonal products)
    p->wg_pack = 1;
    if (f.G > 1 && f.C <= 32 && 64 % f.C == 0 && f.K <= 64 && 64 % f.K == 0 && p->ch.no_pack == 0)
        p->wg_pack = std::min(64 / f.C, 64 / f.K);
    p->wg_cbh = p->wg_pack > 1 ? 1 : (int)cdiv(f.C, 64);
    const int halves = f.taps * p->wg_cbh;
    p->wg_rt = (int)cdiv(halves, 2);
    const int bn_max = p->wg_planes > 1 ? 128 : 256;   // three planes of 256 columns do not fit a stage
    int bn = bn_max;
    for (int c : {256, 128, 64})   // the fewest padded columns, the wider tile on a tie
        if (c <= bn_max && cdiv(f.K, c) * c < cdiv(f.K, bn) * bn) bn = c;
    if (p->wg_pack > 1) bn = 64;
    else if ((p->ch.bn == 64 || p->ch.bn == 128 || p->ch.bn == 256) && p->ch.bn <= bn_max) bn = p->ch.bn;
    p->BN = bn;
    p->wg_nt = p->wg_pack > 1 ? 1 : (int)cdiv(f.K, bn);
    p->wg_nwb = (int)cdiv(f.Wo, 64);
    const int64_t Q = (int64_t)f.N * f.Do * f.Ho * p->wg_nwb;
    if (Q >= ((int64_t)1 << 31)) return false;
    p->wg_q = (int)Q;
    // slab mode (unit stride along W): a unit holds every half of one filter plane in its
    // accumulators and reads one x box per (filter row, channel block) per chunk
    p->wg_slab = 0;
    {
        const int reach = f.dw * (f.X - 1);
        const int hpp = f.Y * f.X * p->wg_cbh;
        const int na = (int)cdiv(hpp, 2);
        if (p->wg_planes == 1 && f.sw == 1 && p->ch.gather != 2 && na <= 8 && na * bn <= 512 && 64 + reach <= 256) {
            const int box_rows = 64 + reach;
            const int box_bytes = (int)cdiv((int64_t)box_rows * 128, 1024) * 1024;
            const int nbox = f.Y * p->wg_cbh;
            const int stage_bytes = nbox * box_bytes + (bn / 64) * 8192;
            const int stages = std::min(8, (int)((232448 - 1024 - 256) / stage_bytes));
            if (stages >= 2) {
                p->wg_slab = 1;
                p->wg_na = na; p->wg_hpp = hpp; p->wg_nbox = nbox; p->wg_box_rows = box_rows;
                p->wg_box_bytes = box_bytes; p->wg_stage_bytes = stage_bytes; p->wg_stages = stages;
                int cols = 32;
                while (cols < na * bn) cols *= 2;
                p->wg_tmem = cols;
            }
        }
    }
    const int64_t base = cdiv(f.G, p->wg_pack) * (p->wg_slab ? f.Z : p->wg_rt) * p->wg_nt;
    if (base >= ((int64_t)1 << 31)) return false;
    int splits = (int)std::max<int64_t>(1, std::min<int64_t>(p->sm_count / base, Q / 2));
    if (p->ch.splits >= 1) splits = (int)std::min<int64_t>(p->ch.splits, Q);
    p->wg_qps = (int)cdiv(Q, splits);
    p->splits = (int)cdiv(Q, p->wg_qps);
    p->total_units = (int)(base * p->splits);
    if ((int64_t)base * p->splits >= ((int64_t)1 << 31)) return false;
    int dev = 0;   // a trial encode checks the boxes against the driver's limits
    if (encode_fn() && cudaGetDevice(&dev) == cudaSuccess && cudaSetDevice(dev) == cudaSuccess) {
        CUtensorMap a, b;
        const void* fake = reinterpret_cast<const void*>((uintptr_t)4096);
        const bool ok = encode_wg_maps(p, fake, fake, &a, &b);
        cudaGetLastError();
        if (!ok) return false;
    }
    cudaGetLastError();
    p->variant = VAR_WG_TC;
    p->prepack_bytes = p->packed_bytes = 0;
    p->workspace_bytes = p->splits > 1 ? (size_t)p->splits * f.G * f.K * f.taps * f.C * sizeof(float) : 0;
    if (p->wg_planes > 1) {   // the workspace also holds the bf16 planes of x and dy
        const size_t nx = (size_t)f.N * f.D * f.H * f.W * f.G * f.C, ndy = (size_t)f.M * f.G * f.K;
        p->wg_xpl_off = align256(p->workspace_bytes);
        p->wg_dypl_off = align256(p->wg_xpl_off + 3 * nx * 2);
        p->workspace_bytes = p->wg_dypl_off + 3 * ndy * 2;
    }
    snprintf(p->desc, sizeof(p->desc),
             "variant=%s direction=bwd_weight operands=%s tile=128x%d row_tiles=%d chunk=64px splits=%d "
             "chunks_per_split=%d units=%d pack=%d",
             p->wg_planes > 1 ? "tc_bf16x3" : "tc_bf16", p->wg_slab ? "mn-major-slab" : "mn-major", bn,
             p->wg_slab ? p->wg_na : p->wg_rt, p->splits, p->wg_qps, p->total_units, p->wg_pack);
    if (p->wg_slab) {
        const size_t n = strlen(p->desc);
        snprintf(p->desc + n, sizeof(p->desc) - n, " boxes=%dx%d stages=%d", p->wg_nbox, p->wg_box_rows, p->wg_stages);
    }
    return true;
}

// Backward weight on the FFMA pipe: 64 x 64 or 128 x 128 tiles of [K] x [taps*C] per group, the output
// pixels split across CTAs until the grid covers the SMs twice (at least one tile width of pixels each).
static void plan_wg_simt(conv_plan* p) {
    const Geom& f = p->fg;
    p->variant = VAR_WG_SIMT;
    // 128 x 128 tiles (8 x 8 per thread) where both extents fill them, else 64 x 64
    p->wg_tile = (f.K >= 96 && (int64_t)f.taps * f.C >= 96) ? 128 : 64;
    p->wg_kt = (int)cdiv(f.K, p->wg_tile);
    p->wg_jt = (int)cdiv((int64_t)f.taps * f.C, p->wg_tile);
    const int64_t tiles = (int64_t)p->wg_kt * p->wg_jt * f.G;
    // at least `tile` pixels per split: shorter splits cost more in partial sums than they gain
    int splits = (int)std::max<int64_t>(1, std::min<int64_t>(2 * p->sm_count / std::max<int64_t>(tiles, 1),
                                                             cdiv(f.M, p->wg_tile)));
    splits = std::min(splits, 64);
    p->wg_mps = (int)(cdiv(cdiv(f.M, splits), 8) * 8);
    p->splits = (int)cdiv(f.M, p->wg_mps);
    p->prepack_bytes = p->packed_bytes = 0;
    p->workspace_bytes = p->splits > 1 ? (size_t)p->splits * f.G * f.K * f.taps * f.C * sizeof(float) : 0;
    snprintf(p->desc, sizeof(p->desc),
             "variant=simt_%s direction=bwd_weight tile=%dx%d pixel_step=8 splits=%d pixels_per_split=%d grid=%dx%dx%d",
             p->dtype == CONV_BF16 ? "bf16" : "f32", p->wg_tile, p->wg_tile, p->splits, p->wg_mps, p->wg_kt, p->wg_jt,
             f.G * p->splits);
}

extern "C" {

conv_status conv_plan_create(conv_plan_t* out, int ndim, int64_t N, int64_t G, int64_t C, int64_t K,
                             const int64_t* spatial, const int64_t* filter, const int64_t* stride,
                             const int64_t* pad, const int64_t* dilation, conv_dtype dtype,
                             conv_epilogue epilogue) {
    if (epilogue < CONV_EPI_NONE || epilogue > CONV_EPI_GELU) return CONV_ERR_INVALID_ARG;
    conv_plan* p = nullptr;
    const conv_status st = init_plan(&p, out, ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype);
    if (st != CONV_OK) return st;
    p->epi = epilogue;
    p->dir = DIR_FWD;
    p->test_stall = env_int("CONV_TEST_STALL", 0) ? 1 : 0;
    // choices: the test hooks if set, else the measured selector's entry for this problem on
    // this device, else the rules
    PlanChoice c;
    if (!choice_from_env(c)) tune_table_lookup(p, c);
    p->ch = c;
    choose_variant(p);
    *out = p;
    return CONV_OK;
}

conv_status conv_bwd_data_plan_create(conv_plan_t* out, int ndim, int64_t N, int64_t G, int64_t C, int64_t K,
                                      const int64_t* spatial, const int64_t* filter, const int64_t* stride,
                                      const int64_t* pad, const int64_t* dilation, conv_dtype dtype) {
    conv_plan* p = nullptr;
    const conv_status st = init_plan(&p, out, ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype);
    if (st != CONV_OK) return st;
    p->epi = CONV_EPI_NONE;
    p->dir = DIR_BWD_DATA;
    const Geom f = p->fg;
    if ((int64_t)f.N * f.D * f.H * f.W >= ((int64_t)1 << 31) - 256 || (int64_t)f.taps * K >= ((int64_t)1 << 30)) {
        delete p;
        return CONV_ERR_UNSUPPORTED;
    }
    // At unit stride dx is the forward convolution of dy with the taps flipped, C and K
    // swapped and padding dil*(F-1) - pad (the transposed convolution), so every forward
    // kernel serves it.  Otherwise each input pixel gathers the dy positions that map onto it.
    const bool transposed = f.sd == 1 && f.sh == 1 && f.sw == 1 && f.dd * (f.Z - 1) >= f.pd &&
                            f.dh * (f.Y - 1) >= f.ph && f.dw * (f.X - 1) >= f.pw;
    choice_from_env(p->ch);   // the test hooks reach every phase's plan too
    if (transposed) {
        Geom& g = p->g;
        g.C = f.K; g.K = f.C;
        g.D = f.Do; g.H = f.Ho; g.W = f.Wo;
        g.pd = f.dd * (f.Z - 1) - f.pd; g.ph = f.dh * (f.Y - 1) - f.ph; g.pw = f.dw * (f.X - 1) - f.pw;
        g.Do = f.D; g.Ho = f.H; g.Wo = f.W;
        g.M = f.N * f.D * f.H * f.W;
        p->Go = g.G; p->Co = g.C; p->Ko = g.K;
        p->dg_fwd = 1;
        p->dg_t0[0] = f.Z - 1; p->dg_t0[1] = f.Y - 1; p->dg_t0[2] = f.X - 1;
        p->dg_dt[0] = p->dg_dt[1] = p->dg_dt[2] = 1;
        PlanChoice c;
        if (!choice_from_env(c)) tune_table_lookup(p, c);
        p->ch = c;
        choose_variant(p);
    } else if (!plan_dg_phased(p)) {
        plan_dg_simt(p);
    }
    *out = p;
    return CONV_OK;
}

conv_status conv_bwd_weight_plan_create(conv_plan_t* out, int ndim, int64_t N, int64_t G, int64_t C, int64_t K,
                                        const int64_t* spatial, const int64_t* filter, const int64_t* stride,
                                        const int64_t* pad, const int64_t* dilation, conv_dtype dtype) {
    conv_plan* p = nullptr;
    const conv_status st = init_plan(&p, out, ndim, N, G, C, K, spatial, filter, stride, pad, dilation, dtype);
    if (st != CONV_OK) return st;
    p->epi = CONV_EPI_NONE;
    p->dir = DIR_BWD_WEIGHT;
    if ((int64_t)G * K * p->g.taps * C >= ((int64_t)1 << 31)) {
        delete p;
        return CONV_ERR_UNSUPPORTED;
    }
    PlanChoice c;
    choice_from_env(c);
    p->ch = c;
    if (!plan_wg_tc(p)) plan_wg_simt(p);
    *out = p;
    return CONV_OK;
}

conv_status conv_plan_output_shape(conv_plan_t plan, int64_t* out_spatial) {
    if (!plan || !out_spatial) return CONV_ERR_INVALID_ARG;
    for (int i = 0; i < plan->ndim; ++i) out_spatial[i] = plan->out_spatial[3 - plan->ndim + i];
    return CONV_OK;
}

size_t conv_prepacked_weight_bytes(conv_plan_t plan) { return plan ? plan->prepack_bytes : 0; }

size_t conv_workspace_bytes(conv_plan_t plan) { return plan ? plan->workspace_bytes : 0; }

conv_status conv_plan_set_workspace(conv_plan_t plan, void* workspace, size_t bytes) {
    if (!plan) return CONV_ERR_INVALID_ARG;
    if (plan->workspace_bytes && (!workspace || bytes < plan->workspace_bytes)) return CONV_ERR_WORKSPACE;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 15u)) return CONV_ERR_ALIGNMENT;
    plan->workspace = workspace;
    plan->workspace_size = bytes;
    return CONV_OK;
}

static bool misaligned(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; }

conv_status conv_prepack_weights(conv_plan_t plan, const void* w, void* w_packed, void* stream) {
    if (!plan || !w || !w_packed) return CONV_ERR_INVALID_ARG;
    if (plan->dir == DIR_BWD_WEIGHT) return CONV_ERR_INVALID_ARG;   // nothing to prepack
    if (misaligned(w) || misaligned(w_packed)) return CONV_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Geom& g = plan->g;
    const int threads = 256;
    if (plan->variant == VAR_DG_SIMT) {
        const Geom& f = plan->fg;
        const long long total = (long long)f.G * plan->Kg * plan->Kpad;
        const int blocks = (int)std::min<long long>(cdiv(total, threads), 65535);
        if (plan->dtype == CONV_BF16)
            prepack_dg_simt_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(
                static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(w_packed), f.K, f.C, f.taps,
                plan->Kg, plan->Kpad, total);
        else
            prepack_dg_simt_kernel<float><<<blocks, threads, 0, s>>>(static_cast<const float*>(w),
                                                                     static_cast<float*>(w_packed), f.K, f.C, f.taps,
                                                                     plan->Kg, plan->Kpad, total);
        return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
    }
    if (plan->variant == VAR_DG_PHASED) {
        for (int i = 0; i < plan->nph; ++i) {
            const conv_status st = conv_prepack_weights(plan->ph[i], w, static_cast<uint8_t*>(w_packed) + plan->ph_off[i],
                                                        stream);
            if (st != CONV_OK) return st;
        }
        return CONV_OK;
    }
    if (plan->dg_fwd) {   // stage the flipped, transposed weight, then prepack it as a forward weight
        const Geom& f = plan->fg;
        void* stage = static_cast<uint8_t*>(w_packed) + plan->dg_src_off;
        TapMap tm;
        tm.Zo = f.Z; tm.Yo = f.Y; tm.Xo = f.X; tm.Zs = g.Z; tm.Ys = g.Y; tm.Xs = g.X;
        for (int i = 0; i < 3; ++i) { tm.t0[i] = plan->dg_t0[i]; tm.dt[i] = plan->dg_dt[i]; }
        const long long total = (long long)f.G * f.K * g.taps * f.C;
        const int blocks = (int)std::min<long long>(cdiv(total, threads), 65535);
        if (plan->dtype == CONV_BF16)
            flip_transpose_kernel<uint16_t><<<blocks, threads, 0, s>>>(static_cast<const uint16_t*>(w),
                                                                      static_cast<uint16_t*>(stage), f.K, f.C, tm, total);
        else
            flip_transpose_kernel<float><<<blocks, threads, 0, s>>>(static_cast<const float*>(w),
                                                                   static_cast<float*>(stage), f.K, f.C, tm, total);
        w = stage;
    }
    if (plan->variant == VAR_TC && plan->tf32) {
        const long long total16 = (long long)(plan->packed_bytes / 32);   // hi and lo written per chunk
        const int blocks = (int)std::min<long long>(cdiv(total16, threads), 65535);
        prepack_tf32x3_kernel<<<blocks, threads, 0, s>>>(static_cast<const float4*>(w), static_cast<uint4*>(w_packed),
                                                         g.K, g.C, g.taps, plan->BN, plan->num_nt, plan->nkb,
                                                         plan->cbt, plan->slab, g.Y, g.X, total16);
    } else if (plan->variant == VAR_TC) {
        const long long total16 = (long long)(plan->packed_bytes / 16);
        const int blocks = (int)std::min<long long>(cdiv(total16, threads), 65535);
        prepack_tc_kernel<<<blocks, threads, 0, s>>>(static_cast<const uint4*>(w), static_cast<uint4*>(w_packed),
                                                     g.K, g.C, g.taps, plan->BN, plan->num_nt, plan->nkb,
                                                     plan->nchunks, plan->cpt, plan->slab ? 2 : plan->tma,
                                                     plan->cbt, plan->pack, plan->Ko, plan->Co, g.Y, g.X, total16);
    } else {
        const long long total = (long long)g.G * plan->Kg * plan->Kpad;
        const int blocks = (int)std::min<long long>(cdiv(total, threads), 65535);
        if (plan->dtype == CONV_BF16)
            prepack_simt_kernel<__nv_bfloat16><<<blocks, threads, 0, s>>>(
                static_cast<const __nv_bfloat16*>(w), static_cast<__nv_bfloat16*>(w_packed), g.K, g.C, g.taps,
                plan->Kg, plan->Kpad, total);
        else
            prepack_simt_kernel<float><<<blocks, threads, 0, s>>>(static_cast<const float*>(w),
                                                                  static_cast<float*>(w_packed), g.K, g.C,
                                                                  g.taps, plan->Kg, plan->Kpad, total);
    }
    return cudaGetLastError() == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

// The split-K reduction: partial sums in split order, then the epilogue.
static conv_status launch_reduce_n(conv_plan_t plan, const float* ws, const void* bias, void* y, long long MGK,
                                   int GK, int epi, cudaStream_t s, const Lattice& lat = Lattice{}) {
    const Geom& g = plan->g;
    const int threads = 256;
    const long long work = GK % 4 == 0 ? MGK / 4 : MGK;
    const int blocks = (int)std::min<long long>(cdiv(work, threads), (long long)plan->sm_count * 8);
    const bool pdl = plan->overlap != 0;
    cudaError_t e;
    if (plan->dtype == CONV_BF16)
        e = launch_kernel(splitk_reduce_kernel<__nv_bfloat16>, dim3(blocks), dim3(threads), 0, s, pdl, 1, ws,
                          plan->splits, MGK, GK, static_cast<const __nv_bfloat16*>(bias),
                          static_cast<__nv_bfloat16*>(y), epi, (int)pdl, lat, g.Do, g.Ho, g.Wo);
    else
        e = launch_kernel(splitk_reduce_kernel<float>, dim3(blocks), dim3(threads), 0, s, pdl, 1, ws, plan->splits, MGK,
                          GK, static_cast<const float*>(bias), static_cast<float*>(y), epi, (int)pdl, lat, g.Do, g.Ho,
                          g.Wo);
    return e == cudaSuccess ? CONV_OK : CONV_ERR_CUDA;
}

static conv_status launch_reduce(conv_plan_t plan, const float* ws, const void* bias, void* y, cudaStream_t s) {
    const Geom& g = plan->g;
    return launch_reduce_n(plan, ws, bias, y, (long long)g.M * g.G * g.K, g.G * g.K, (int)plan->epi, s, plan->lat);
}

// Argument checks shared by both forward entry points.
static conv_status check_forward_args(conv_plan_t plan, const void* x, const void* w_packed, const void* bias,
                                      const void* y) {
    if (!plan || !x || !w_packed || !y) return CONV_ERR_INVALID_ARG;
    if (plan->dir != DIR_FWD) return CONV_ERR_INVALID_ARG;
    const bool needs_bias = plan->epi == CONV_EPI_BIAS || plan->epi == CONV_EPI_BIAS_GELU;
    if (needs_bias && !bias) return CONV_ERR_INVALID_ARG;
    if (misaligned(x) || misaligned(w_packed) || misaligned(y) || (needs_bias && misaligned(bias)))
        return CONV_ERR_ALIGNMENT;
    return CONV_OK;
}

// Enqueue the forward pass with ws as the split-K workspace (null when the plan has none).
static conv_status run_forward(conv_plan_t plan, const void* x, const void* w_packed, const void* bias, void* y,
                               float* ws, cudaStream_t s) {
    const bool needs_bias = plan->epi == CONV_EPI_BIAS || plan->epi == CONV_EPI_BIAS_GELU;
    unsigned* err = error_word_ptr();
    if (!err) return CONV_ERR_CUDA;
    cudaError_t e;
    if (plan->variant == VAR_TC) {
        TcParams tp;
        tp.g = plan->g;
        tp.x = x; tp.wpack = w_packed; tp.bias = needs_bias ? bias : nullptr; tp.y = y;
        tp.ws = ws;
        tp.err = err;
        tp.BN = plan->BN; tp.num_mt = plan->num_mt; tp.num_nt = plan->num_nt; tp.nkb = plan->nkb;
        tp.nchunks = plan->nchunks; tp.cpt = plan->cpt; tp.splits = plan->splits; tp.kbps = plan->kbps;
        tp.epi = (int)plan->epi; tp.total_units = plan->total_units;
        tp.tma = plan->tma; tp.map_kind = plan->map_kind; tp.BW = plan->BW; tp.BH = plan->BH;
        tp.tiles_w = plan->tiles_w; tp.tiles_h = plan->tiles_h; tp.cbt = plan->cbt; tp.tf32 = plan->tf32;
        tp.sleep_mask = plan->sleep_mask;
        tp.slab = plan->slab; tp.slab_bws = plan->slab_bws; tp.slab_hr = plan->slab_hr; tp.slab_nkg = plan->slab_nkg;
        tp.slab_nbg = plan->slab_nbg; tp.slab_btaps = plan->slab_btaps; tp.slab_sa = plan->slab_sa;
        tp.slab_sb = plan->slab_sb; tp.slab_a_stage = plan->slab_a_stage; tp.slab_resident = plan->slab_resident;
        tp.slab_nacc = plan->slab ? plan->slab_nacc : 1; tp.slab_pair_rows = plan->slab_pair_rows;
        tp.acc_bh = plan->slab ? plan->acc_bh : plan->BH;
        tp.pdl = plan->overlap;
        tp.epi_warps = plan->epi_warps ? plan->epi_warps : 8;
        tp.cluster_red = plan->cluster_red;
        tp.mc = plan->tma && !plan->slab ? plan->mc : 0;
        // outputs land on the plan's lattice only where the kernel writes final values; partial
        // sums (split-K through the reduction kernel) are indexed by GEMM row
        const bool partial = plan->splits > 1 && !plan->cluster_red;
        tp.lat = (plan->lat.on && !partial) ? plan->lat : identity_lattice(plan->g.Do, plan->g.Ho, plan->g.Wo);
        tp.test_stall = plan->test_stall;
        tp.f_splits = make_fastdiv(plan->splits); tp.f_num_nt = make_fastdiv(plan->num_nt);
        tp.f_G = make_fastdiv(plan->g.G); tp.f_tiles_w = make_fastdiv(plan->tiles_w);
        tp.f_tiles_h = make_fastdiv(plan->tiles_h); tp.f_Do = make_fastdiv(plan->g.Do);
        tp.f_Ho = make_fastdiv(plan->g.Ho); tp.f_Wo = make_fastdiv(plan->g.Wo); tp.f_cbt = make_fastdiv(plan->cbt);
        tp.f_cpt = make_fastdiv(plan->cpt); tp.f_X = make_fastdiv(plan->g.X);
        tp.f_YX = make_fastdiv(plan->g.Y * plan->g.X); tp.f_BW = make_fastdiv(plan->BW);
        tp.f_bws = make_fastdiv(plan->slab_bws);
        CUtensorMap map, ymap;
        if (plan->tma && !encode_act_map(plan, x, &map)) return CONV_ERR_CUDA;
        tp.ystore = plan->ystore && !tp.lat.on;
        if (tp.ystore && !encode_y_map(plan, y, &ymap)) return CONV_ERR_CUDA;
        if (plan->pair) {
            CUtensorMap wmap;
            if (!encode_w_map(plan, w_packed, &wmap)) return CONV_ERR_CUDA;
            e = plan->slab ? launch_slab_pair(tp, &map, &wmap, plan->grid, plan->slab_smem, s)
                           : launch_pair(tp, &map, &wmap, tp.ystore ? &ymap : nullptr, plan->stages, plan->grid, s);
        } else {
            e = plan->slab ? launch_slab(tp, &map, plan->grid, plan->slab_smem, s)
                           : launch_tc(tp, plan->tma ? &map : nullptr, tp.ystore ? &ymap : nullptr, plan->stages,
                                       plan->grid, s);
        }
    } else {
        SimtParams sp;
        sp.g = plan->g;
        sp.x = x; sp.wpack = w_packed; sp.bias = needs_bias ? bias : nullptr; sp.y = y;
        sp.ws = ws;
        sp.dg = 0; sp.rows = plan->g.M; sp.cols = plan->g.K; sp.rch = plan->g.C;
        sp.Kg = plan->Kg; sp.Kpad = plan->Kpad; sp.num_mt = plan->num_mt; sp.num_nt = plan->num_nt;
        sp.nkt = plan->nkt; sp.splits = plan->splits; sp.ktps = plan->ktps; sp.epi = (int)plan->epi;
        sp.pdl = plan->overlap;
        e = launch_simt(sp, plan->dtype == CONV_BF16, plan->BM, plan->vec != 0, s);
    }
    if (e != cudaSuccess) return CONV_ERR_CUDA;
    if (plan->splits > 1 && !plan->cluster_red) return launch_reduce(plan, ws, needs_bias ? bias : nullptr, y, s);
    return CONV_OK;
}

conv_status conv_fwd(conv_plan_t plan, const void* x, const void* w_packed, const void* bias, void* y,
                     void* stream) {
    const conv_status st = check_forward_args(plan, x, w_packed, bias, y);
    if (st != CONV_OK) return st;
    if (plan->workspace_bytes && (!plan->workspace || plan->workspace_size < plan->workspace_bytes))
        return CONV_ERR_WORKSPACE;
    return run_forward(plan, x, w_packed, bias, y, static_cast<float*>(plan->workspace),
                       static_cast<cudaStream_t>(stream));
}

conv_status conv_plan_set_overlap(conv_plan_t plan, int enable) {
    if (!plan) return CONV_ERR_INVALID_ARG;
    plan->overlap = enable ? 1 : 0;
    return CONV_OK;
}

// A plan's workspace, or null; CONV_ERR_WORKSPACE when it needs one that is missing.
static conv_status plan_workspace(conv_plan_t plan, float** ws) {
    if (plan->workspace_bytes && (!plan->workspace || plan->workspace_size < plan->workspace_bytes))
        return CONV_ERR_WORKSPACE;
    *ws = plan->workspace_bytes ? static_cast<float*>(plan->workspace) : nullptr;
    return CONV_OK;
}

conv_status conv_bwd_data(conv_plan_t plan, const void* dy, const void* w_packed, void* dx, void* stream) {
    if (!plan || !dy || !w_packed || !dx || plan->dir != DIR_BWD_DATA) return CONV_ERR_INVALID_ARG;
    if (misaligned(dy) || misaligned(w_packed) || misaligned(dx)) return CONV_ERR_ALIGNMENT;
    float* ws = nullptr;
    const conv_status st = plan_workspace(plan, &ws);
    if (st != CONV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (plan->dg_fwd) return run_forward(plan, dy, w_packed, nullptr, dx, ws, s);
    if (plan->variant == VAR_DG_PHASED) {
        const Geom& f = plan->fg;
        if (plan->ph_zero &&
            cudaMemsetAsync(dx, 0, (size_t)f.N * f.D * f.H * f.W * f.G * f.C * (plan->dtype == CONV_BF16 ? 2 : 4), s) !=
                cudaSuccess)
            return CONV_ERR_CUDA;
        for (int i = 0; i < plan->nph; ++i) {
            conv_plan* q = plan->ph[i];
            // phases write disjoint pixels of dx: each may overlap the one before it
            q->overlap = (i > 0 || (plan->overlap && !plan->ph_zero)) ? 1 : 0;
            const conv_status st = run_forward(q, dy, static_cast<const uint8_t*>(w_packed) + plan->ph_off[i], nullptr,
                                               dx, ws, s);
            if (st != CONV_OK) return st;
        }
        return CONV_OK;
    }
    const Geom& f = plan->fg;
    SimtParams sp;
    sp.g = f;
    sp.x = dy; sp.wpack = w_packed; sp.bias = nullptr; sp.y = dx; sp.ws = ws;
    sp.dg = 1; sp.rows = f.N * f.D * f.H * f.W; sp.cols = f.C; sp.rch = f.K;
    sp.Kg = plan->Kg; sp.Kpad = plan->Kpad; sp.num_mt = plan->num_mt; sp.num_nt = plan->num_nt;
    sp.nkt = plan->nkt; sp.splits = plan->splits; sp.ktps = plan->ktps; sp.epi = EPI_NONE;
    sp.pdl = plan->overlap;
    if (launch_simt(sp, plan->dtype == CONV_BF16, plan->BM, plan->vec != 0, s) != cudaSuccess) return CONV_ERR_CUDA;
    if (plan->splits > 1)
        return launch_reduce_n(plan, ws, nullptr, dx, (long long)sp.rows * f.G * f.C, f.G * f.C, EPI_NONE, s);
    return CONV_OK;
}

conv_status conv_bwd_weight(conv_plan_t plan, const void* x, const void* dy, void* dw, void* stream) {
    if (!plan || !x || !dy || !dw || plan->dir != DIR_BWD_WEIGHT) return CONV_ERR_INVALID_ARG;
    if (misaligned(x) || misaligned(dy) || misaligned(dw)) return CONV_ERR_ALIGNMENT;
    float* ws = nullptr;
    const conv_status st = plan_workspace(plan, &ws);
    if (st != CONV_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const Geom& f = plan->fg;
    if (plan->variant == VAR_WG_TC) {
        unsigned* err = error_word_ptr();
        if (!err) return CONV_ERR_CUDA;
        const void* xs = x;
        const void* dys = dy;
        if (plan->wg_planes > 1) {   // fp32: split x and dy into their bf16 planes first
            uint8_t* wsb = reinterpret_cast<uint8_t*>(plan->workspace);
            const long long nx = (long long)f.N * f.D * f.H * f.W * f.G * f.C, ndy = (long long)f.M * f.G * f.K;
            __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(wsb + plan->wg_xpl_off);
            __nv_bfloat16* dyp = reinterpret_cast<__nv_bfloat16*>(wsb + plan->wg_dypl_off);
            const int threads = 256;
            split_planes_kernel<<<(int)std::min<long long>(cdiv(nx, threads), (long long)plan->sm_count * 8), threads, 0, s>>>(
                static_cast<const float*>(x), xp, nx);
            split_planes_kernel<<<(int)std::min<long long>(cdiv(ndy, threads), (long long)plan->sm_count * 8), threads, 0,
                                  s>>>(static_cast<const float*>(dy), dyp, ndy);
            if (cudaGetLastError() != cudaSuccess) return CONV_ERR_CUDA;
            xs = xp;
            dys = dyp;
        }
        CUtensorMap xm, dym;
        if (!encode_wg_maps(plan, xs, dys, &xm, &dym)) return CONV_ERR_CUDA;
        WgradTcParams tp;
        tp.g = f;
        tp.dw = dw; tp.ws = ws; tp.err = err;
        tp.BN = plan->BN; tp.RT = plan->wg_rt; tp.NT = plan->wg_nt;
        tp.splits = plan->splits; tp.Q = plan->wg_q; tp.qps = plan->wg_qps; tp.nwb = plan->wg_nwb;
        tp.cbh = plan->wg_cbh; tp.halves = f.taps * plan->wg_cbh; tp.total_units = plan->total_units;
        tp.pack = plan->wg_pack;
        tp.planes = plan->wg_planes;
        tp.slab = plan->wg_slab; tp.na = plan->wg_na; tp.hpp = plan->wg_hpp; tp.nbox = plan->wg_nbox;
        tp.box_rows = plan->wg_box_rows; tp.box_bytes = plan->wg_box_bytes; tp.stage_bytes = plan->wg_stage_bytes;
        tp.stages = plan->wg_stages; tp.tmem_cols = plan->wg_tmem;
        tp.pdl = plan->overlap;
        if (launch_wgrad_tc(tp, &xm, &dym, s) != cudaSuccess) return CONV_ERR_CUDA;
        if (plan->splits > 1)
            return launch_reduce_n(plan, ws, nullptr, dw, (long long)f.G * f.K * f.taps * f.C, f.taps * f.C, EPI_NONE,
                                   s);
        return CONV_OK;
    }
    WgradParams wp;
    wp.g = f;
    wp.x = x; wp.dy = dy; wp.dw = dw; wp.ws = ws;
    wp.tile = plan->wg_tile;
    wp.num_kt = plan->wg_kt; wp.num_jt = plan->wg_jt; wp.splits = plan->splits; wp.mps = plan->wg_mps;
    wp.pdl = plan->overlap;
    if (launch_wgrad_simt(wp, plan->dtype == CONV_BF16, s) != cudaSuccess) return CONV_ERR_CUDA;
    if (plan->splits > 1) {
        const long long n = (long long)f.G * f.K * f.taps * f.C;
        return launch_reduce_n(plan, ws, nullptr, dw, n, f.taps * f.C, EPI_NONE, s);
    }
    return CONV_OK;
}

conv_status conv_plan_check(conv_plan_t plan, void* stream) {
    if (!plan) return CONV_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return CONV_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) return CONV_ERR_CUDA;
    if (v) {
        const unsigned zero = 0;
        if (cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero)) != cudaSuccess) return CONV_ERR_CUDA;
        return CONV_ERR_TIMEOUT;
    }
    return CONV_OK;
}

conv_status conv_plan_destroy(conv_plan_t plan) {
    if (plan)
        for (int i = 0; i < plan->nph; ++i) delete plan->ph[i];
    delete plan;
    return CONV_OK;
}

const char* conv_status_string(conv_status status) {
    switch (status) {
        case CONV_OK: return "CONV_OK";
        case CONV_ERR_INVALID_ARG: return "CONV_ERR_INVALID_ARG";
        case CONV_ERR_UNSUPPORTED: return "CONV_ERR_UNSUPPORTED";
        case CONV_ERR_ALIGNMENT: return "CONV_ERR_ALIGNMENT";
        case CONV_ERR_WORKSPACE: return "CONV_ERR_WORKSPACE";
        case CONV_ERR_CUDA: return "CONV_ERR_CUDA";
        case CONV_ERR_TIMEOUT: return "CONV_ERR_TIMEOUT";
    }
    return "CONV_ERR_UNKNOWN";
}

const char* conv_plan_describe(conv_plan_t plan) { return plan ? plan->desc : ""; }

}  // extern "C"

// ----------------------------------------------------------------------------- allocation-free forward
// Split-K partial sums in a file-scope device array, for callers that cannot allocate
// device memory (see conv_fwd_static_scratch in conv.h).
namespace {
__device__ __align__(256) float g_static_scratch[CONV_STATIC_SCRATCH_BYTES / sizeof(float)];

std::mutex g_scratch_mu;
float* g_scratch_ptr[64];

// Device address of the array on the current device, looked up once per device.
float* static_scratch_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = static_cast<float*>(p);
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" conv_status conv_fwd_static_scratch(conv_plan_t plan, const void* x, const void* w_packed,
                                               const void* bias, void* y, void* stream) {
    const conv_status st = check_forward_args(plan, x, w_packed, bias, y);
    if (st != CONV_OK) return st;
    if (plan->workspace_bytes > CONV_STATIC_SCRATCH_BYTES) return CONV_ERR_WORKSPACE;
    float* scratch = nullptr;
    if (plan->workspace_bytes) {
        scratch = static_scratch_ptr();
        if (!scratch) return CONV_ERR_CUDA;
    }
    return run_forward(plan, x, w_packed, bias, y, scratch, static_cast<cudaStream_t>(stream));
}

extern "C" {

size_t conv_static_scratch_bytes(void) { return sizeof(g_static_scratch); }

double conv_plan_flops(conv_plan_t plan) { return plan ? plan->flops : 0.0; }

}  // extern "C"

// ----------------------------------------------------------------------------- measured selector: entry points
extern "C" {

size_t conv_tune_scratch_bytes(conv_plan_t plan) {
    if (!plan || plan->dir == DIR_BWD_WEIGHT || (plan->dir == DIR_BWD_DATA && !plan->dg_fwd)) return 0;
    size_t need = 0;
    for (const conv_plan& t : tune_candidates(plan)) need = std::max(need, align256(t.prepack_bytes) + t.workspace_bytes);
    return need;
}

conv_status conv_plan_tune(conv_plan_t plan, const void* x, const void* w, const void* bias, void* y, void* scratch,
                           size_t scratch_bytes, int iters, void* stream) {
    if (!plan || !x || !w || !y || !scratch || iters < 1) return CONV_ERR_INVALID_ARG;
    if (plan->dir == DIR_BWD_WEIGHT || (plan->dir == DIR_BWD_DATA && !plan->dg_fwd)) return CONV_ERR_UNSUPPORTED;
    const bool needs_bias = plan->epi == CONV_EPI_BIAS || plan->epi == CONV_EPI_BIAS_GELU;
    if (needs_bias && !bias) return CONV_ERR_INVALID_ARG;
    if (misaligned(x) || misaligned(w) || misaligned(y) || misaligned(scratch) || (needs_bias && misaligned(bias)))
        return CONV_ERR_ALIGNMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::vector<conv_plan> cands = tune_candidates(plan);
    cudaEvent_t e0, e1;
    if (cudaEventCreate(&e0) != cudaSuccess) return CONV_ERR_CUDA;
    if (cudaEventCreate(&e1) != cudaSuccess) {
        cudaEventDestroy(e0);
        return CONV_ERR_CUDA;
    }
    float best = 0.0f;
    int best_i = -1;
    std::vector<std::pair<std::string, double>> log;
    conv_status st = CONV_OK;
    for (size_t i = 0; i < cands.size() && st == CONV_OK; ++i) {
        conv_plan& t = cands[i];
        const size_t wbytes = align256(t.prepack_bytes);
        if (wbytes + t.workspace_bytes > scratch_bytes) continue;
        uint8_t* wp = static_cast<uint8_t*>(scratch);
        float* ws = t.workspace_bytes ? reinterpret_cast<float*>(wp + wbytes) : nullptr;
        if (conv_prepack_weights(&t, w, wp, stream) != CONV_OK) continue;
        bool ok = true;
        for (int r = 0; r < 2 && ok; ++r) ok = run_forward(&t, x, wp, bias, y, ws, s) == CONV_OK;
        ok = ok && cudaEventRecord(e0, s) == cudaSuccess;
        for (int r = 0; r < iters && ok; ++r) ok = run_forward(&t, x, wp, bias, y, ws, s) == CONV_OK;
        ok = ok && cudaEventRecord(e1, s) == cudaSuccess;
        if (cudaStreamSynchronize(s) != cudaSuccess) {   // a failed launch leaves the context unusable
            st = CONV_ERR_CUDA;
            break;
        }
        // a candidate whose kernels gave up on a wait is not taken
        unsigned v = 0;
        if (cudaMemcpyFromSymbol(&v, g_error_word, sizeof(v)) != cudaSuccess) {
            st = CONV_ERR_CUDA;
            break;
        }
        if (v) {
            const unsigned zero = 0;
            cudaMemcpyToSymbol(g_error_word, &zero, sizeof(zero));
            ok = false;
        }
        float ms = 0.0f;
        if (ok && cudaEventElapsedTime(&ms, e0, e1) == cudaSuccess) {
            log.emplace_back(t.desc, 1e3 * ms / iters);
            if (best_i < 0 || ms < best) {
                best = ms;
                best_i = (int)i;
            }
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    if (st != CONV_OK) return st;
    if (best_i < 0) return CONV_ERR_WORKSPACE;   // no candidate fitted the scratch buffer
    const PlanChoice bc = cands[best_i].ch;
    {
        std::lock_guard<std::mutex> lk(g_tune_mu);
        TuneEntry& e = g_tune_table[plan_key(plan)];
        e.c = bc;
        e.us = 1e3 * best / iters;
        e.log = std::move(log);
    }
    plan->ch = bc;
    choose_variant(plan);
    return CONV_OK;
}

conv_status conv_tune_table_save(const char* path) {
    if (!path) return CONV_ERR_INVALID_ARG;
    FILE* f = fopen(path, "w");
    if (!f) return CONV_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lk(g_tune_mu);
    for (const auto& kv : g_tune_table) {
        const PlanChoice& c = kv.second.c;
        fprintf(f, "%s | simt=%d no_pack=%d bn=%d bm=%d splits=%d gather=%d slab_stream=%d slab_pair=%d epi_warps=%d "
                   "cluster_red=%d mc=%d pair=%d",
                kv.first.c_str(), c.simt, c.no_pack, c.bn, c.bm, c.splits, c.gather, c.slab_stream, c.slab_pair,
                c.epi_warps, c.cluster_red, c.mc, c.pair);
        if (kv.second.us >= 0.0) fprintf(f, " | us=%.3f", kv.second.us);
        fputc('\n', f);
        // the measurements behind the choice, as comment lines (ignored by the loader)
        for (const auto& r : kv.second.log) fprintf(f, "#\tus=%.3f\t%s\n", r.second, r.first.c_str());
    }
    const bool ok = fclose(f) == 0;
    return ok ? CONV_OK : CONV_ERR_INVALID_ARG;
}

conv_status conv_tune_table_load(const char* path) {
    if (!path) return CONV_ERR_INVALID_ARG;
    FILE* f = fopen(path, "r");
    if (!f) return CONV_ERR_INVALID_ARG;
    char line[1024];
    conv_status st = CONV_OK;
    std::vector<std::pair<std::string, TuneEntry>> rows;
    while (fgets(line, sizeof(line), f)) {
        if (line[0] == '\n' || line[0] == '#') continue;
        char* bar = strstr(line, " | ");
        TuneEntry te;
        PlanChoice& c = te.c;
        // (rows written before the mc and pair fields existed carry ten or eleven fields: the
        // missing ones stay with the rules)
        int nf = bar ? sscanf(bar + 3,
                              "simt=%d no_pack=%d bn=%d bm=%d splits=%d gather=%d slab_stream=%d slab_pair=%d "
                              "epi_warps=%d cluster_red=%d mc=%d pair=%d",
                              &c.simt, &c.no_pack, &c.bn, &c.bm, &c.splits, &c.gather, &c.slab_stream, &c.slab_pair,
                              &c.epi_warps, &c.cluster_red, &c.mc, &c.pair)
                     : 0;
        if (nf < 10 || nf > 12) {
            st = CONV_ERR_INVALID_ARG;
            break;
        }
        if (const char* u = strstr(bar + 3, " | us=")) te.us = atof(u + 6);
        rows.emplace_back(std::string(line, bar - line), te);
    }
    fclose(f);
    if (st != CONV_OK) return st;   // a malformed file changes nothing
    std::lock_guard<std::mutex> lk(g_tune_mu);
    for (auto& r : rows) g_tune_table[r.first] = r.second;
    return CONV_OK;
}

conv_status conv_tune_table_clear(void) {
    std::lock_guard<std::mutex> lk(g_tune_mu);
    g_tune_table.clear();
    return CONV_OK;
}

}  // extern "C"
