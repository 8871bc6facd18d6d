// Backward weight of the grouped convolution on the FFMA pipe (the "bwd_weight" variant
// that page "composable_kernel dispatcher/heuristics/LEARNINGS_GROUPED_CONV.md",
// section 6, names for the NHWGC / GKYXC / NHWGK layouts):
//
//   dw[g][k][tap][c] = sum over output pixels m of dy[m][g][k] * x[source(m, tap)][g][c]
//
// with source(m, tap) = o*stride - pad + tap*dil per spatial dimension (zero outside the
// input).  Per group this is a GEMM whose rows are the K output channels, whose columns
// j = tap*C + c run over the filter, and whose reduction runs over the output pixels.
//
// CTA tile TK (k) x TJ (j) = 64 x 64 or 128 x 128, 8 pixels per step, 256 threads each holding
// a (TK/16) x (TJ/16) block; double-buffered shared memory with register prefetch.  The pixels are split across
// CTAs (blockIdx.z = group * splits + split); with more than one split each writes fp32
// partials that the split-K reduction sums in split order.
#include <cuda_bf16.h>
#include <stdint.h>

#include "internal.h"

namespace convfwd {
namespace {

constexpr int BKM = 8, THREADS = 256;

__device__ __forceinline__ float ldf(const float* p) { return __ldg(p); }
__device__ __forceinline__ float ldf(const __nv_bfloat16* p) { return __bfloat162float(p[0]); }
__device__ __forceinline__ void stf(float* p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T, int TK, int TJ>
__global__ void __launch_bounds__(THREADS) conv_wgrad_simt_kernel(const __grid_constant__ WgradParams p) {
    if (p.pdl) {
        griddep_launch();
        griddep_wait();
    }
    constexpr int RK = TK / 16, RJ = TJ / 16;      // per-thread block
    constexpr int LQ = TK / 32;                    // values each thread loads per step (A and B)
    __shared__ __align__(16) float As[2][BKM][TK + 4];   // dy values  [pixel][k]
    __shared__ __align__(16) float Bs[2][BKM][TJ + 4];   // x gathered [pixel][j]
    const Geom& g = p.g;
    const T* x = reinterpret_cast<const T*>(p.x);
    const T* dy = reinterpret_cast<const T*>(p.dy);
    const int tid = threadIdx.x;
    const int k0 = blockIdx.x * TK, j0 = blockIdx.y * TJ;
    const int gi = blockIdx.z / p.splits, split = blockIdx.z % p.splits;
    const int M = g.M;
    const int m0 = split * p.mps;
    const int m1 = min(m0 + p.mps, M);
    const int NJ = g.taps * g.C;
    const int GK = g.G * g.K, GC = g.G * g.C;

    // loader slots: pixel row lm of the step, LQ consecutive k (A) and LQ consecutive j (B)
    const int lm = tid >> 5;
    const int lq = (tid & 31) * LQ;
    int jz[LQ], jy[LQ], jx[LQ], jc[LQ];
    bool jok[LQ];
#pragma unroll
    for (int e = 0; e < LQ; ++e) {
        const int j = j0 + lq + e;
        jok[e] = j < NJ;
        const int tap = jok[e] ? j / g.C : 0;
        jc[e] = jok[e] ? j - tap * g.C : 0;
        jz[e] = tap / (g.Y * g.X);
        const int r = tap - jz[e] * g.Y * g.X;
        jy[e] = r / g.X;
        jx[e] = r - jy[e] * g.X;
    }
    float ra[LQ], rb[LQ];
    auto load_step = [&](int mb) {
        const int m = mb + lm;
#pragma unroll
        for (int e = 0; e < LQ; ++e) ra[e] = rb[e] = 0.f;
        if (m >= m1) return;
        int t = m;
        const int ow = t % g.Wo; t /= g.Wo;
        const int oh = t % g.Ho; t /= g.Ho;
        const int od = t % g.Do;
        const int n = t / g.Do;
        const T* dyp = dy + (long long)m * GK + (long long)gi * g.K;
#pragma unroll
        for (int e = 0; e < LQ; ++e)
            if (k0 + lq + e < g.K) ra[e] = ldf(dyp + k0 + lq + e);
#pragma unroll
        for (int e = 0; e < LQ; ++e) {
            if (!jok[e]) continue;
            const int id = od * g.sd - g.pd + jz[e] * g.dd;
            const int ih = oh * g.sh - g.ph + jy[e] * g.dh;
            const int iw = ow * g.sw - g.pw + jx[e] * g.dw;
            if ((unsigned)id >= (unsigned)g.D || (unsigned)ih >= (unsigned)g.H || (unsigned)iw >= (unsigned)g.W)
                continue;
            rb[e] = ldf(x + ((((long long)n * g.D + id) * g.H + ih) * g.W + iw) * GC + (long long)gi * g.C + jc[e]);
        }
    };
    auto store_step = [&](int buf) {
#pragma unroll
        for (int e = 0; e < LQ; ++e) {
            As[buf][lm][lq + e] = ra[e];
            Bs[buf][lm][lq + e] = rb[e];
        }
    };

    float acc[RK][RJ];
#pragma unroll
    for (int i = 0; i < RK; ++i)
#pragma unroll
        for (int j = 0; j < RJ; ++j) acc[i][j] = 0.f;
    const int ty = tid >> 4, tx = tid & 15;   // rows k0 + RK ty.., columns j0 + RJ tx..
    if (m0 < m1) {
        load_step(m0);
        store_step(0);
        __syncthreads();
        int buf = 0;
        for (int mb = m0; mb < m1; mb += BKM) {
            const bool more = mb + BKM < m1;
            if (more) load_step(mb + BKM);
#pragma unroll
            for (int q = 0; q < BKM; ++q) {
                float av[RK], bv[RJ];
#pragma unroll
                for (int i = 0; i < RK; i += 4) {
                    const float4 a = *reinterpret_cast<const float4*>(&As[buf][q][ty * RK + i]);
                    av[i] = a.x; av[i + 1] = a.y; av[i + 2] = a.z; av[i + 3] = a.w;
                }
#pragma unroll
                for (int j = 0; j < RJ; j += 4) {
                    const float4 b = *reinterpret_cast<const float4*>(&Bs[buf][q][tx * RJ + j]);
                    bv[j] = b.x; bv[j + 1] = b.y; bv[j + 2] = b.z; bv[j + 3] = b.w;
                }
#pragma unroll
                for (int i = 0; i < RK; ++i)
#pragma unroll
                    for (int j = 0; j < RJ; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
            }
            if (more) store_step(buf ^ 1);
            __syncthreads();
            buf ^= 1;
        }
    }
    // dw (or the partials) [G][K][taps*C]
#pragma unroll
    for (int i = 0; i < RK; ++i) {
        const int k = k0 + ty * RK + i;
        if (k >= g.K) continue;
        const long long row = ((long long)gi * g.K + k) * NJ;
#pragma unroll
        for (int j = 0; j < RJ; ++j) {
            const int jj = j0 + tx * RJ + j;
            if (jj >= NJ) continue;
            if (p.splits > 1)
                p.ws[(long long)split * g.G * g.K * NJ + row + jj] = acc[i][j];
            else
                stf(reinterpret_cast<T*>(p.dw) + row + jj, acc[i][j]);
        }
    }
}

}  // namespace

cudaError_t launch_wgrad_simt(const WgradParams& p, bool bf16, cudaStream_t stream) {
    dim3 grid(p.num_kt, p.num_jt, p.g.G * p.splits);
    if (p.tile == 128)
        return bf16 ? launch_kernel(conv_wgrad_simt_kernel<__nv_bfloat16, 128, 128>, grid, dim3(THREADS), 0, stream,
                                    p.pdl != 0, 1, p)
                    : launch_kernel(conv_wgrad_simt_kernel<float, 128, 128>, grid, dim3(THREADS), 0, stream, p.pdl != 0,
                                    1, p);
    return bf16 ? launch_kernel(conv_wgrad_simt_kernel<__nv_bfloat16, 64, 64>, grid, dim3(THREADS), 0, stream,
                                p.pdl != 0, 1, p)
                : launch_kernel(conv_wgrad_simt_kernel<float, 64, 64>, grid, dim3(THREADS), 0, stream, p.pdl != 0, 1, p);
}

}  // namespace convfwd
