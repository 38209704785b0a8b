// wq_internal.h -- internal declarations shared by the host API and the kernel launchers.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

#include "../../include/wq.h"

namespace wq {

constexpr int kBlockM = 128;        // GEMM tile rows (tcgen05 M)
constexpr int kBlockN = 128;        // GEMM tile columns (tcgen05 N)
constexpr int kStageK = 256;        // K elements per pipeline stage (128 bytes of fp4)
constexpr int kSfAtom = 512;        // bytes of one 128-row x 64-K block-scale atom

// Device-side layout of one activation workspace for M rows.
struct ActWorkspace {
    uint8_t* codes = nullptr;       // [M, K/2]
    uint8_t* sf = nullptr;          // MMA layout, ceil(M/128) * K/64 atoms
    float* g = nullptr;             // [M]
    uint16_t* u = nullptr;          // [M, r] bf16 (r: stored rank)
    uint16_t* xo = nullptr;         // [M, n_out] fp16 (n_out: stored width)
    unsigned int* amax = nullptr;   // batch maximum of WQ_ACT_SCALE_TENSOR (fp32 bits)
    size_t bytes = 0;
};

// r and n_out are the stored widths (side_width of the configured counts).
ActWorkspace carve_workspace(void* base, int M, int K, int r, int n_out);

// Stored width of a 16-bit side operand (U columns, x_O columns): 0, 16, 32 or 64, the widths
// the tcgen05 side MMAs and the 32/64/128-byte swizzled TMA boxes take; the columns beyond the
// configured count hold zeros.
inline int side_width(int n) { return n == 0 ? 0 : (n <= 16 ? 16 : (n <= 32 ? 32 : 64)); }

// Schedule knobs (tests and tuning): taken from the environment once, at first use, and changed
// afterwards only through wq_set_tuning.  -1 (or 0 where stated) means "choose automatically".
enum TuneKnob {
    kTuneFused = 0,        // WQ_FUSED: 1 = the fused small-batch kernel where it applies
    kTuneGemmSplit,        // WQ_GEMM_SPLIT: CTAs per output tile of the single-CTA GEMM (0 = auto)
    kTuneGemmWide,         // WQ_GEMM_WIDE: 1 / 0 pins the CTA-pair GEMM on / off
    kTuneGemmPush,         // WQ_GEMM_PUSH: 0 = pull form of the split-K reduction
    kTuneGemmStages,       // WQ_GEMM_STAGES: ring depth cap of the single-CTA GEMM (0 = auto)
    kTuneQuantSchedule,    // WQ_QUANT_SCHEDULE: 1 = stream, 0 = cluster (or "stream" / "cluster")
    kTuneQuantSplit,       // WQ_QUANT_SPLIT: CTAs per row tile of the cluster quantiser (0 = auto)
    kTuneQuantCtasPerSm,   // WQ_QUANT_CTAS_PER_SM: resident stream-quantiser CTAs per SM (0 = auto)
    kTuneGemmDb,           // WQ_GEMM_DB: 1 / 0 pins the two-accumulator form of the pair GEMM on / off
    kTuneCount
};
int tune(TuneKnob k);

struct QuantArgs {
    const void* x;                  // bf16 [M, K]
    const CUtensorMap* tmX;         // x as [M, K] bf16, box 64 x 16, swizzle 128B
    const uint32_t* pfrag;          // P in mma.sync B-fragment order (see wq_api.cu)
    int* err;                       // device error flag
    int M, K;
    const float* inv_s;             // [K] or null; per 32-channel half, pairs (s_k, s_k+16), k = 0..15
    const float* inv_s_rr = nullptr;// the same [K] with per 64-block the pairs (s_k, s_k+32), k = 0..31
    int rotate;
    const uint32_t* omega_blk;      // [K/64][4]: kept-channel mask (lo, hi), x_O index of the first, 0
    int n_out;                      // kept channels (0: none)
    int xo_ld;                      // row stride of x_O in elements (>= n_out; the columns beyond are zeroed)
    uint16_t* xo;                   // fp16 [M, xo_ld]
    const uint16_t* P;              // bf16 [K, r]
    int r;                          // stored rank (0, 16, 32 or 64); U columns beyond the rank are 0
    uint16_t* u;                    // bf16 [M, r]
    uint8_t* codes;                 // [M, K/2]
    uint8_t* sf;                    // scales, layout per `sf_layout`
    int sf_layout;                  // WQ_SCALE_LAYOUT_*
    float* g;                       // [M]
    int num_sms;                    // used to spread small batches over more CTAs
    bool int8 = false;              // 8-bit layer: codes are int8 values stored as bf16 [M, K]
    bool fp8 = false;               // with int8: e4m3 bytes [M, K] instead, scale amax / 448
    bool fp8_bf16 = false;          // with fp8: the e4m3 values as exact bf16 [M, K] (W4A8)
    const uint16_t* vt = nullptr;   // Q-WAM projected complement: bf16 [r_real, K] (null: off)
    int r_real = 0;                 // the configured rank (the projection's loop length)
    // Activation tensor scale: WQ_ACT_SCALE_ROW (one per row, from the row), WQ_ACT_SCALE_TENSOR
    // (one for all M rows: a first launch takes the maximum, a second quantises) or
    // WQ_ACT_SCALE_STATIC (the calibrated `static_g`, one pass).  Every mode writes g[m] per row.
    int act_scale = WQ_ACT_SCALE_ROW;
    float static_g = 0.0f;
    unsigned int* amax_bits = nullptr;  // WQ_ACT_SCALE_TENSOR: running maximum (fp32 bits), zeroed by the caller
};

cudaError_t launch_quantize_act(const QuantArgs& a, cudaStream_t stream);
// True when M rows take a persistent schedule (stream or register-resident; else the cluster
// schedule).
bool quant_stream_schedule(int M, int num_sms);
// The register-resident schedule (wq_quant_rr.cu): 4-bit layers, per-row scales, K <= 1536.
bool quant_resident_eligible(const QuantArgs& a);
cudaError_t launch_quantize_resident(const QuantArgs& a, cudaStream_t stream);

// The epilogue quantises the tile's bf16 output for the next layer instead of storing it
// (wq_linear_forward_chain): the next layer's smoothing, block-64 FWHT along this layer's N, kept
// channels and NVFP4 coding with its fixed tensor scale.
struct ChainArgs {
    const float* inv_s;             // next layer's inv_s in pair order [N] or null
    int rotate;                     // bit 0: FWHT; bit 1: smooth after the rotation
    const uint32_t* omega_blk;      // next layer's kept-channel table [N/64][4] or null
    int n_out, xo_ld;               // kept channels and the x_O row stride
    uint16_t* xo;                   // fp16 [M, xo_ld]
    uint8_t* codes;                 // [M, N/2]
    uint8_t* sf;                    // MMA layout, ceil(M/128) x N/64 atoms
    float* g_out;                   // [M], every entry the fixed g
    float g;                        // the next layer's fixed tensor scale
};

struct GemmArgs {
    int M, N, K, r, n_out;
    const CUtensorMap* tmA;   // activation codes [M, K/2] u8, box 128x128, swizzle 128B
    const CUtensorMap* tmB;   // weight codes     [N, K/2] u8, box 128x128, swizzle 128B
    const CUtensorMap* tmU;   // U      [M, r]     bf16, box r x 128
    const CUtensorMap* tmQ;   // Q^T    [N, r]     bf16, box r x 128
    const CUtensorMap* tmXO;  // x_O    [M, n_out] fp16, box n_out x 128
    const CUtensorMap* tmWO;  // W_O^T  [N, n_out] fp16, box n_out x 128
    const CUtensorMap* tmY;   // y      [M, N]     bf16, box 64 x 32, swizzle 128B
    // the scales as [128-row blocks][K/64 blocks][128 u32] (one 512-byte atom per row block and
    // K block), boxes of 4 K blocks x 1 (activations) or 2 (weights) row blocks; CTA-pair schedule
    const CUtensorMap* tmSFA = nullptr;
    const CUtensorMap* tmSFB = nullptr;
    // the two-accumulator pair schedule (256 x 192 tiles): this CTA's 96 rows of the weight codes,
    // Q^T and W_O^T; the weight scales in 192-row tile layout (two atoms per tile and K block,
    // rows 128..191 in the second); y in 32 x 32 boxes without swizzle
    const CUtensorMap* tmB96 = nullptr;
    const CUtensorMap* tmQ96 = nullptr;
    const CUtensorMap* tmWO96 = nullptr;
    const CUtensorMap* tmSFB192 = nullptr;
    const CUtensorMap* tmY32 = nullptr;
    const uint8_t* sfa;       // activation scales, MMA layout
    const uint8_t* sfb;       // weight scales, MMA layout
    const float* gA;          // [M]
    float gW;
    const float* bias;        // [N] or null
    int* err;                 // device error flag
    int num_sms;
    void* y;                  // bf16 [M, N] (written directly by the split-K reduction)
    int force_split;          // 0: choose; otherwise CTAs per tile (power of two <= 16)
    bool w8 = false;          // 8-bit layer: A/W are int8 codes stored as bf16 [., K] (or e4m3, fp8)
    bool fp8 = false;         // 8-bit layer with e4m3 bytes [., K] (kind::f8f6f4)
    const float* colscale = nullptr;  // 8-bit layer: per-output-column scale [N]
    const ChainArgs* chain = nullptr; // non-null: quantise the output for the next layer (pair schedule)
};

cudaError_t launch_gemm(const GemmArgs& a, cudaStream_t stream);
// 0: 128 x 128 tiles on persistent single CTAs; 1: split-K clusters; 2: 256 x 256 tiles on CTA
// pairs; -1 on a CUDA error.  Only the shape, mode, SM count and force_split of `a` are read.
int gemm_schedule(const GemmArgs& a);
// CTA-pair schedule (256 x 256 tiles) for batches with many output tiles (wq_gemm2.cu).
cudaError_t launch_gemm_wide(const GemmArgs& a, cudaStream_t stream);
int wide_gemm_tiles(int M, int N);
// Two-accumulator CTA-pair schedule (256 x 192 tiles, wq_gemm3.cu): 4-bit layers, no chain.
cudaError_t launch_gemm_wide_db(const GemmArgs& a, cudaStream_t stream);
int wide_db_tiles(int M, int N);

// The whole W4A4 forward of a small batch in one kernel (wq_fused.cu).
struct FusedArgs {
    int M, K, N, r, n_out;
    int nb, cs;                     // 64-blocks per CTA, CTAs per cluster (from fused_plan)
    const CUtensorMap* tmX;         // x [M, K] bf16, box 64 x 16, swizzle 128B
    const CUtensorMap* tmB;         // weight codes, box (32 nb bytes) x 128, swizzle of that width
    const CUtensorMap* tmQ;         // Q^T    [N, r]     bf16, box r x 128
    const CUtensorMap* tmWO;        // W_O^T  [N, n_out] fp16, box n_out x 128
    const float* inv_s;             // pair order, or null
    int rotate;
    const uint32_t* omega_blk;
    const uint32_t* pfrag;
    const uint8_t* sfb;             // weight scales, MMA layout
    float gW;
    const float* bias;
    void* y;                        // bf16 [M, N]
    int* err;
};

bool fused_plan(int M, int K, int N, int r, int n_out, int& nb, int& cs);
cudaError_t launch_fused(const FusedArgs& a, cudaStream_t stream);

struct ConvArgs {
    const void* x;            // bf16 NCDHW [B, C, D, H, W]
    int C, D, H, W, V, N;     // V = B D H W voxels over the batch, N output channels
    float* partial;           // [2 num_sms] per-CTA maxima of |x|
    float* g;                 // tensor scale of the input
    uint8_t* codes;           // [V, C/2]
    uint8_t* scales;          // [V, C/16]
    const CUtensorMap* tmB;   // weight codes [N, 27 C / 2] u8, box 64 x 128, swizzle 64B
    const uint8_t* sfb;       // weight scales, MMA layout
    float gw;
    void* y;                  // bf16 NCDHW [B, N, D, H, W]
    int* err;
    int num_sms;
};

size_t conv_workspace_bytes(int C, int V, int num_sms);
cudaError_t launch_conv_quant(const ConvArgs& a, cudaStream_t stream);
cudaError_t launch_conv_gemm(const ConvArgs& a, cudaStream_t stream);

// Record a message for wq_last_error() (thread-local).
void set_last_error(const char* msg);

// The device a handle's memory lives on (the device current at its preparation).
int handle_device(wq_weights_t h);

// cuTensorMapEncodeTiled obtained from the driver at run time (no libcuda link).
bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                    uint64_t outer, uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer,
                    CUtensorMapSwizzle swizzle, const char** why);
// The MMA-layout scales of `rows` rows and K columns as a 3-D map: [row blocks][K/64][128 u32],
// boxes of 4 K blocks x box_row_blocks row blocks (out-of-range atoms read as zeros).
bool encode_scale_tmap(CUtensorMap* map, const void* base, int rows, int K, int box_row_blocks, const char** why);
// The same over an explicit number of 128-row atom blocks (the weights' 192-row tile layout).
bool encode_scale_tmap_blocks(CUtensorMap* map, const void* base, int row_blocks, int K, int box_row_blocks,
                              const char** why);

}  // namespace wq
