// Internal definitions shared by the library's translation units (not installed).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

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

// Device error word codes (bit flags).
enum : unsigned { ERR_WAIT_TIMEOUT = 1u };

// ---- tensor-core (tcgen05) bf16 implicit GEMM ----
struct TcParams {
    Geom g;
    const void* x;          // bf16 N D H W G C
    const void* wpack;      // swizzled tiles [G][NT][NKB][BN x 128 B]
    const void* bias;       // bf16 G*K or null
    void* y;                // bf16 N Do Ho Wo G K
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
};

// Launch the tensor-core kernel for a (BN, stages) pair chosen by the plan.
cudaError_t launch_tc_bf16(const TcParams& p, int stages, int grid, cudaStream_t stream);
size_t tc_smem_bytes(int BN, int stages);
bool tc_config_supported(int BN, int stages);

// ---- SIMT FFMA implicit GEMM (fp32 I/O; also bf16 where channel counts rule out the tensor path) ----
struct SimtParams {
    Geom g;
    const void* x;          // T  N D H W G C
    const void* wpack;      // T  [G][taps*C][Kpad]
    const void* bias;       // T  G*K or null
    void* y;                // T  N Do Ho Wo G K
    float* ws;              // split-K partials [splits][M][G*K]
    int Kg;                 // taps*C
    int Kpad;               // K rounded up to the N tile
    int num_mt, num_nt;
    int nkt;                // K steps of 8 along Kg
    int splits, ktps;       // split-K factor, K steps per split
    int epi;
};

cudaError_t launch_simt(const SimtParams& p, bool bf16, int BM, bool vec, cudaStream_t stream);

}  // namespace convfwd
