// Internal definitions shared by the library's translation units (not installed).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

namespace convfwd {

// A problem in the 3-spatial form (conv1d: D = H = 1, conv2d: D = 1), channels last.
struct Geom {
    int N, D, H, W, G, C, K;
    int Z, Y, X;
    int sd, sh, sw;     // stride
    int pd, ph, pw;     // padding (both sides)
    int dd, dh, dw;     // dilation
    int Do, Ho, Wo;
    int M;              // N*Do*Ho*Wo output pixels (GEMM M per group)
    int taps;           // Z*Y*X
};

enum Epi { EPI_NONE = 0, EPI_BIAS = 1, EPI_BIAS_GELU = 2, EPI_GELU = 3 };

// Division by a divisor fixed at plan time, done by a multiplication (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994, the round-up
// method): with s = ceil(log2 d) and m = floor(2^32 (2^s - d) / d) + 1,
// floor(n / d) = (mulhi(n, m) + n) >> s for every 0 <= n < 2^31.  The kernels' per-tile
// index arithmetic (unit -> tile -> pixel) runs on these instead of hardware-less integer
// division sequences, which cost a few hundred cycles each on the first tile.
struct FastDiv {
    uint32_t d, m, s;
};
inline FastDiv make_fastdiv(uint32_t d) {
    FastDiv f;
    f.d = d < 1 ? 1 : d;
    uint32_t s = 0;
    while (s < 31 && (1ull << s) < f.d) ++s;
    f.s = s;
    f.m = (uint32_t)((((1ull << s) - f.d) << 32) / f.d + 1);
    return f;
}
#ifdef __CUDACC__
__device__ __forceinline__ int fdiv(int n, const FastDiv& f) {
    return (int)((__umulhi((uint32_t)n, f.m) + (uint32_t)n) >> f.s);
}
#endif

#ifdef __CUDACC__
// Programmatic dependent launch.  griddep_launch: this CTA allows the next kernel on the
// stream (if launched as a programmatic dependent) to start; griddep_wait: block until the
// kernel before this one on the stream has completed and its writes are visible.  Every
// thread that reads data a previous kernel may produce (x, bias) or writes data it may
// still read (y, workspace) calls griddep_wait first.
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

// Launch a kernel, as a programmatic dependent of the previous kernel on the stream when
// pdl is set; with cluster_x > 1, as thread-block clusters of cluster_x consecutive CTAs.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 bool pdl, int cluster_x, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (pdl) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (cluster_x > 1) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = (unsigned)cluster_x;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = n ? attr : nullptr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Device error word codes (bit flags).
enum : unsigned { ERR_WAIT_TIMEOUT = 1u };

// Output placement.  Normally output pixel (n, od, oh, ow) is row ((n*Do + od)*Ho + oh)*Wo + ow
// of y.  With on = 1 the outputs are a lattice of a larger tensor of D x H x W pixels: pixel
// (n, od, oh, ow) goes to (n, r_d + s_d*od, r_h + s_h*oh, r_w + s_w*ow) there (one stride phase
// of a backward-data pass).
struct Lattice {
    int on;
    int D, H, W;
    int sd, sh, sw;
    int rd, rh, rw;
};

// The identity placement of a problem whose output extents are Do x Ho x Wo (on = 0: the
// kernels may still evaluate lattice_pixel with it, which gives the plain NDHW row).
inline Lattice identity_lattice(int Do, int Ho, int Wo) {
    Lattice L;
    L.on = 0;
    L.D = Do; L.H = Ho; L.W = Wo;
    L.sd = L.sh = L.sw = 1;
    L.rd = L.rh = L.rw = 0;
    return L;
}

// (pixel indices of every tensor the plans accept stay below 2^31, so 32-bit arithmetic)
__host__ __device__ __forceinline__ int lattice_pixel(const Lattice& L, int n, int od, int oh, int ow) {
    return ((n * L.D + L.rd + L.sd * od) * L.H + L.rh + L.sh * oh) * L.W + L.rw + L.sw * ow;
}

// ---- tensor-core (tcgen05) bf16 implicit GEMM ----
struct TcParams {
    Geom g;
    const void* x;          // bf16 or fp32, N D H W G C
    const void* wpack;      // swizzled tiles [G][NT][NKB][BN x 128 B] (3xTF32: hi tile then lo tile)
    const void* bias;       // G*K of the I/O type, or null
    void* y;                // N Do Ho Wo G K of the I/O type
    float* ws;              // split-K partials [splits][M][G*K] fp32 (splits > 1)
    unsigned* err;          // device error word
    int BN;                 // N tile (output channels per CTA tile)
    int num_mt, num_nt;     // tiles along M and N
    int nkb;                // 64-wide K blocks per group (taps*C padded to 64)
    int nchunks;            // taps*C/8 (16-byte chunks along K)
    int cpt;                // C/8 chunks per tap
    int splits, kbps;       // split-K factor and K blocks per split
    int epi;
    int total_units;        // num_mt*G*num_nt*splits
    // TMA gather: one tiled-tensor load per K block of a BH x BW block of output pixels
    // (one (n, od) plane) for one tap and one 64-channel block.
    int tma;                // 1: TMA gather, 0: cp.async gather
    int map_kind;           // 0: tensor dims {G*C, W, H, D, N}; 1: {C, G, W, H, N} (D = Z = 1)
    int BW, BH;             // output tile extent along W and H (BW*BH <= 128 rows)
    int tiles_w, tiles_h;   // tiles per output plane
    int cbt;                // channel blocks per tap (64 bf16 or 32 fp32 channels; kb = tap*cbt + block)
    int tf32;               // 1: fp32 I/O as 3xTF32 (TMA gather only)
    int sleep_mask;         // which roles wait with a suspend hint: 1 producer, 2 epilogue, 4 MMA
    // slab mode (stride 1): one box of HR input rows x BWs pixels per (tile, input plane,
    // channel block) serves all Y*X taps of that plane as row-shifted windows
    int slab;               // 1: slab mode (always with tma = 1)
    int slab_bws;           // slab row pitch in pixels: BW + dw*(X-1)
    int slab_hr;            // slab rows: BH + dh*(Y-1)
    int slab_nkg;           // k-groups per tile: Z * cbt (input plane, channel block)
    int slab_nbg;           // weight ring stages per k-group (filter rows Y)
    int slab_btaps;         // taps per weight stage (filter columns X)
    int slab_sa, slab_sb;   // slab ring and weight ring stages (resident: weight chunks held)
    int slab_resident;      // 1: the weights of one (group, N tile) stay in shared memory
    int slab_nacc;          // accumulators per unit: 1, or 2 (two tiles stacked along H)
    int slab_pair_rows;     // slab row of the second accumulator's windows (acc_bh * BWs)
    int acc_bh;             // output rows per accumulator (BH / slab_nacc)
    int slab_a_stage;       // bytes per slab stage (3xTF32: hi half then lo half)
    int pdl;                // 1: launched as a programmatic dependent (see griddep_wait)
    int epi_warps;          // per-tap kernel: 8 or 16 epilogue warps
    int cluster_red;        // 1: the splits of a tile run as one cluster and sum their partial
                            // accumulators through distributed shared memory (no workspace)
    int mc;                 // 1 (per-tap bf16 TMA kernel, no split): CTA pairs share each weight tile
                            // by multicast; units are pairs of M tiles (see conv_fwd_tc_kernel)
    int ystore;             // 1: the epilogue stores y through a tensor map (TMA), one 64-channel x
                            // 32-pixel box per warp and chunk (tiles of one output row, BW % 32 == 0)
    Lattice lat;            // where the output pixels land in y (one phase of a strided backward data)
    int test_stall;         // test hook: the MMA role waits on a barrier nothing completes
    // divisors of the per-tile index arithmetic
    FastDiv f_splits, f_num_nt, f_G, f_tiles_w, f_tiles_h, f_Do, f_Ho, f_Wo, f_cbt, f_cpt, f_X, f_YX, f_BW, f_bws;
};

constexpr size_t SLAB_SMEM_MAX = 232448;   // dynamic shared memory a block may opt in to

// Output columns one epilogue warp of the per-tap kernels (one CTA or a pair) stages and stores
// at a time for bf16 outputs: its columns, up to 64 (a 128-byte row segment).  (Chunks of 32
// for 256-wide tiles with 16 epilogue warps would halve their staging and make room for a
// fourth ring stage: measured no faster, since the three producer warps keep three stages in
// flight either way.)
__host__ __device__ constexpr int tc_store_cols(int bn, int ew, bool pair) {
    return (void)pair, (bn / (ew / 4) < 64 ? bn / (ew / 4) : 64);
}

// Launch the tensor-core kernel for the (BN, stages) pair the plan picked (see tc_stages_for).
cudaError_t launch_tc(const TcParams& p, const CUtensorMap* act_map, const CUtensorMap* y_map, int stages, int grid,
                      cudaStream_t stream);
int tc_stages_for(int BN, int tf32, int epi_warps);
// Clusters of two CTAs of the weight-multicast kernel for (BN, epi_warps) that can be resident at
// once on the current device (0 if it cannot be queried).
int tc_mc_max_clusters(int BN, int epi_warps);
// CTA-pair kernel (tc_pair.cu): M = 256 tiles over two CTAs with .cta_group::2 MMAs; bf16 per-tap
// TMA plans without a split.  w_map: the packed weights as 2-D rows of 128 bytes, boxes of BN/2 rows.
cudaError_t launch_pair(const TcParams& p, const CUtensorMap* act_map, const CUtensorMap* w_map,
                        const CUtensorMap* y_map, int stages, int grid, cudaStream_t stream);
int tc_pair_stages_for(int BN, int epi_warps);
int tc_pair_max_clusters(int BN, int epi_warps);
// Slab kernel on CTA pairs (tc_slab_pair.cu): bf16 tile-pair slab plans (two accumulators per
// unit), N tiles of 32 or 64; each CTA holds half of every weight tile (w_map as for launch_pair).
cudaError_t launch_slab_pair(const TcParams& p, const CUtensorMap* act_map, const CUtensorMap* w_map, int grid,
                             size_t smem, cudaStream_t stream);
size_t slab_pair_smem_bytes(int BN, int sa, int sb, size_t a_stage, int btaps);
int slab_pair_max_clusters(size_t smem);
// Slab-mode kernel; smem from slab_smem_bytes.
cudaError_t launch_slab(const TcParams& p, const CUtensorMap* act_map, int grid, size_t smem, cudaStream_t stream);
size_t slab_smem_bytes(int BN, int tf32, int sa, int sb, size_t a_stage, int btaps);

// ---- SIMT FFMA implicit GEMM (fp32 I/O; also bf16 where channel counts rule out the tensor path) ----
// Forward: GEMM rows are output pixels (N Do Ho Wo), columns the K output channels of a
// group, the reduction index tap*C + c.  Backward data (dg = 1): rows are input pixels
// (N D H W), columns the C input channels, the reduction index tap*K + k over dy, whose
// source position per tap is (i + pad - tap*dil) / stride where that division is exact.
struct SimtParams {
    Geom g;                 // the forward problem
    const void* x;          // T  forward: x (N D H W G C); backward data: dy (N Do Ho Wo G K)
    const void* wpack;      // T  [G][taps*rch][Kpad]
    const void* bias;       // T  G*K or null
    void* y;                // T  forward: y (N Do Ho Wo G K); backward data: dx (N D H W G C)
    float* ws;              // split-K partials [splits][rows][G*cols]
    int dg;                 // 1: backward data
    int rows, cols, rch;    // GEMM rows, columns per group, reduction channels per tap
    int Kg;                 // taps*rch
    int Kpad;               // cols rounded up to the N tile
    int num_mt, num_nt;
    int nkt;                // K steps of 8 along Kg
    int splits, ktps;       // split-K factor, K steps per split
    int epi;
    int pdl;
};

cudaError_t launch_simt(const SimtParams& p, bool bf16, int BM, bool vec, cudaStream_t stream);

// ---- backward weight ----
// dw[g][k][tap][c] = sum over output pixels m of dy[m][g][k] * x[source of m at tap][g][c].
// FFMA kernel: per CTA a 64 (k) x 64 (tap*C + c) tile of one group over a range of output
// pixels; with splits > 1 each split writes fp32 partials [splits][G][K][taps*C].
struct WgradParams {
    Geom g;
    const void* x;          // T  N D H W G C
    const void* dy;         // T  N Do Ho Wo G K
    void* dw;               // T  G K taps C (splits == 1)
    float* ws;              // partials (splits > 1)
    int tile;               // 64 (64 x 64 tiles) or 128 (128 x 128)
    int num_kt, num_jt;     // tiles along K and along taps*C
    int splits, mps;        // pixel splits, pixels per split
    int pdl;
};
cudaError_t launch_wgrad_simt(const WgradParams& p, bool bf16, cudaStream_t stream);

// Tensor-core backward weight (bf16): per group, D[(tap, c)][k] accumulates x * dy over output
// pixels, both operands read by TMA in their own channels-last layouts and fed to tcgen05.mma
// as MN-major tiles.  Rows: pairs of 64-channel "halves" h = tap * cbh + cb (2 per 128-row
// tile); columns: BN output channels; reduction: chunks of 64 pixels along one output row.
struct WgradTcParams {
    Geom g;
    void* dw;               // bf16 G K taps C (splits == 1)
    float* ws;              // fp32 partials [splits][G][K][taps*C] (splits > 1)
    unsigned* err;
    int BN, RT, NT;         // N tile, row tiles, column tiles
    int splits, Q, qps;     // pixel splits, 64-pixel chunks in all, chunks per split
    int nwb;                // 64-pixel blocks per output row
    int cbh, halves;        // 64-channel blocks per tap, taps * cbh
    // slab mode (unit stride along W): a unit covers every half of one filter plane z
    int slab;               // 1: slab mode
    int na;                 // accumulators per unit (halves of a plane / 2, rounded up)
    int hpp;                // halves per filter plane: Y * X * cbh
    int nbox;               // x boxes per chunk: Y * cbh, each box_rows pixels of 64 channels
    int box_rows, box_bytes, stage_bytes, stages;
    int tmem_cols;
    int planes;             // 1: bf16 x and dy; 3: fp32 split into hi, mid, lo bf16 planes (images
                            // pl*N + n of the plane tensors), dw in fp32
    int pack;               // groups per tile (C, K dividing 64): x rows and dy columns of `pack`
                            // consecutive groups share one box; only the diagonal blocks are kept
    int total_units;
    int pdl;
};
cudaError_t launch_wgrad_tc(const WgradTcParams& p, const CUtensorMap* xmap, const CUtensorMap* dymap,
                            cudaStream_t stream);

}  // namespace convfwd
