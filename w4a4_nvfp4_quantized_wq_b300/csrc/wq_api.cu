// wq_api.cu -- the C ABI declared in include/wq.h: argument checks, offline weight folding
// and NVFP4 quantisation (host, fp64 fold), device residency of the prepared weights,
// tensor-map construction and the two-kernel forward.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>
#include <vector>

#include "wq_internal.h"

namespace {

thread_local std::string g_last_error;

wq_status fail(wq_status s, const std::string& msg) {
    g_last_error = msg;
    return s;
}

wq_status cuda_fail(cudaError_t e, const char* what) {
    return fail(WQ_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define WQ_CUDA(call, what)                                  \
    do {                                                     \
        cudaError_t e_ = (call);                             \
        if (e_ != cudaSuccess) return cuda_fail(e_, what);   \
    } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

uint16_t bf16_bits(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// bf16 of an fp64 value with one rounding to nearest even: first to fp32 rounding to odd (truncate,
// then set the last bit when anything was cut off), which keeps the information a later
// round-to-nearest at 8 bits needs, then fp32 -> bf16 round-to-nearest-even.
uint16_t bf16_bits_from_f64(double v) {
    float t = static_cast<float>(v);                      // nearest
    if (static_cast<double>(t) != v && std::isfinite(t)) {
        if (std::fabs(static_cast<double>(t)) > std::fabs(v)) t = std::nextafter(t, 0.0f);   // toward zero
        uint32_t u;
        std::memcpy(&u, &t, 4);
        u |= 1u;                                          // sticky: inexact
        std::memcpy(&t, &u, 4);
    }
    return bf16_bits(t);
}
uint16_t f16_bits(float f) { return __half_as_ushort(__float2half_rn(f)); }

float e4m3_value(uint32_t c) {
    const uint32_t e = (c >> 3) & 15u, m = c & 7u;
    if (e == 0) return static_cast<float>(m) * 0.001953125f;
    return std::ldexp(1.0f + static_cast<float>(m) / 8.0f, static_cast<int>(e) - 7);
}

// In-place block-64 Walsh-Hadamard transform (fp64) of a strided vector: butterflies at
// strides 1, 2, 4, 8, 16, 32, then the 1/8 normalisation.
void fwht64_f64(double* v, size_t stride) {
    for (int h = 1; h < 64; h <<= 1)
        for (int i = 0; i < 64; ++i)
            if ((i & h) == 0) {
                const double a = v[i * stride], b = v[(i + h) * stride];
                v[i * stride] = a + b;
                v[(i + h) * stride] = a - b;
            }
    for (int i = 0; i < 64; ++i) v[i * stride] = v[i * stride] * 0.125;
}

template <typename F>
void parallel_for(size_t n, F&& f) {
    unsigned nt = std::max(1u, std::min(32u, std::thread::hardware_concurrency()));
    if (n < 64) nt = 1;
    std::vector<std::thread> th;
    const size_t chunk = (n + nt - 1) / nt;
    for (unsigned t = 0; t < nt; ++t) {
        const size_t lo = t * chunk, hi = std::min(n, lo + chunk);
        if (lo >= hi) break;
        th.emplace_back([&f, lo, hi] { for (size_t i = lo; i < hi; ++i) f(i); });
    }
    for (auto& x : th) x.join();
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

CUtensorMapSwizzle swizzle_for_row_bytes(uint32_t b) {
    return b == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : (b == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}

}  // namespace

namespace wq {

void set_last_error(const char* msg) { g_last_error = msg; }

namespace {
struct KnobDef {
    const char* name;
    int dflt;
};
constexpr KnobDef kKnobs[kTuneCount] = {
    {"WQ_FUSED", 0},          {"WQ_GEMM_SPLIT", 0},     {"WQ_GEMM_WIDE", -1},        {"WQ_GEMM_PUSH", -1},
    {"WQ_GEMM_STAGES", 0},    {"WQ_QUANT_SCHEDULE", -1}, {"WQ_QUANT_SPLIT", 0},      {"WQ_QUANT_CTAS_PER_SM", 0},
    {"WQ_GEMM_DB", -1},
};
std::once_flag g_knob_once;
}  // namespace
std::atomic<int> g_knob[kTuneCount];
namespace {

// The environment is read once; afterwards only wq_set_tuning changes a knob.
void init_knobs() {
    std::call_once(g_knob_once, [] {
        for (int k = 0; k < kTuneCount; ++k) {
            int v = kKnobs[k].dflt;
            if (const char* e = std::getenv(kKnobs[k].name)) {
                if (k == kTuneQuantSchedule && (e[0] == 's' || e[0] == 'c' || e[0] == 'r'))
                    v = e[0] == 's' ? 1 : (e[0] == 'r' ? 2 : 0);
                else if (e[0] != '\0')
                    v = std::atoi(e);
            }
            g_knob[k].store(v, std::memory_order_relaxed);
        }
    });
}

int knob_index(const char* name) {
    if (!name) return -1;
    for (int k = 0; k < kTuneCount; ++k)
        if (std::strcmp(name, kKnobs[k].name) == 0) return k;
    return -1;
}
}  // namespace

int tune(TuneKnob k) {
    init_knobs();
    return g_knob[k].load(std::memory_order_relaxed);
}

bool encode_tmap_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner, uint64_t outer,
                    uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swizzle,
                    const char** why) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) { *why = "cuTensorMapEncodeTiled unavailable"; return false; }
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { *why = "cuTensorMapEncodeTiled failed"; return false; }
    return true;
}

bool encode_scale_tmap(CUtensorMap* map, const void* base, int rows, int K, int box_row_blocks, const char** why) {
    return encode_scale_tmap_blocks(map, base, (rows + kBlockM - 1) / kBlockM, K, box_row_blocks, why);
}

bool encode_scale_tmap_blocks(CUtensorMap* map, const void* base, int row_blocks, int K, int box_row_blocks,
                              const char** why) {
    EncodeTiledFn fn = get_encode_fn();
    if (!fn) { *why = "cuTensorMapEncodeTiled unavailable"; return false; }
    const uint64_t nkb = static_cast<uint64_t>(K / 64);
    const cuuint64_t dims[3] = {kSfAtom / 4, nkb, static_cast<cuuint64_t>(row_blocks)};
    const cuuint64_t strides[2] = {kSfAtom, nkb * kSfAtom};
    const cuuint32_t box[3] = {kSfAtom / 4, 4, static_cast<cuuint32_t>(box_row_blocks)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) { *why = "cuTensorMapEncodeTiled failed (scales)"; return false; }
    return true;
}

ActWorkspace carve_workspace(void* base, int M, int K, int r, int n_out) {
    ActWorkspace w;
    const size_t m_pad = align_up(static_cast<size_t>(M), kBlockM);
    size_t off = 0;
    auto take = [&](size_t bytes) { const size_t o = off; off = align_up(off + bytes, 1024); return o; };
    const size_t o_codes = take(static_cast<size_t>(M) * K / 2);
    const size_t o_sf = take(m_pad / kBlockM * (K / 64) * kSfAtom);
    const size_t o_g = take(static_cast<size_t>(M) * 4);
    const size_t o_u = take(static_cast<size_t>(M) * r * 2);
    const size_t o_xo = take(static_cast<size_t>(M) * n_out * 2);
    const size_t o_amax = take(16);
    w.bytes = off;
    if (base) {
        uint8_t* b = static_cast<uint8_t*>(base);
        w.codes = b + o_codes;
        w.sf = b + o_sf;
        w.g = reinterpret_cast<float*>(b + o_g);
        w.u = reinterpret_cast<uint16_t*>(b + o_u);
        w.xo = reinterpret_cast<uint16_t*>(b + o_xo);
        w.amax = reinterpret_cast<unsigned int*>(b + o_amax);
    }
    return w;
}

}  // namespace wq

struct wq_weights {
    wq_config cfg{};
    int device = 0;
    int num_sms = 0;
    float gW = 0.0f;
    uint8_t* d_codes = nullptr;    // [N, K/2]
    uint8_t* d_sf = nullptr;       // MMA layout, ceil(N/128) * K/64 atoms
    float* d_bias = nullptr;       // [N]
    float* d_inv_s = nullptr;      // [K], quantiser pair order (see pair_order)
    float* d_inv_s_rr = nullptr;   // [K], per 64-block the pairs (k, k + 32) (register-resident quantiser)
    uint32_t* d_omega_blk = nullptr;// [K/64][4]: Omega bit mask (2 words), index of its first channel, 0
    uint16_t* d_P = nullptr;       // [K, r] bf16
    uint32_t* d_Pfrag = nullptr;   // P in mma.sync m16n8k16 B-fragment order
    uint16_t* d_Qt = nullptr;      // [N, r] bf16
    uint16_t* d_WOt = nullptr;     // [N, n_out] fp16
    int* d_err = nullptr;
    float* d_colscale = nullptr;   // W8A8: per-output-column weight scale [N]
    uint16_t* d_wexp = nullptr;    // W4A8: the NVFP4 weight values (code x block scale) as exact bf16 [N, K]
    uint16_t* d_Vt = nullptr;      // projected complement: bf16 [rank, K], the protected subspace's basis
    int r_pad = 0;                 // stored rank: side_width(rank) (U, P, Q^T columns)
    int no_pad = 0;                // stored outlier width: side_width(n_outliers) (x_O, W_O^T columns)
    unsigned int* d_amax = nullptr;// WQ_ACT_SCALE_TENSOR: running batch maximum of wq_quantize_activations
    int conv_cin = 0;              // Conv3d handles: input channels (K = 27 conv_cin)
    CUtensorMap tmBconv{};         // weight codes with 64-byte boxes (Conv3d, fused small-batch path)
    CUtensorMap tmB{}, tmQ{}, tmWO{};
    CUtensorMap tmSFB{};           // weight scales in 4-K-block x 2-row-block boxes (CTA-pair GEMM)
    // two-accumulator pair GEMM (256 x 192 tiles): 96-row boxes of the weight codes, Q^T and W_O^T,
    // and the weight scales in 192-row tile layout (two atoms per tile and K block)
    uint8_t* d_sf192 = nullptr;
    CUtensorMap tmB96{}, tmQ96{}, tmWO96{}, tmSFB192{};
    // activation / output tensor maps, re-encoded when the buffers change
    std::mutex mu;
    const void* key_codes = nullptr;
    const void* key_u = nullptr;
    const void* key_xo = nullptr;
    const void* key_y = nullptr;
    const void* key_sf = nullptr;
    int key_M = -1;
    CUtensorMap tmA{}, tmU{}, tmXO{}, tmY{}, tmSFA{}, tmY32{};
    std::mutex mu_x;
    const void* key_x = nullptr;
    int key_xM = -1;
    CUtensorMap tmX{};
    // host-buffer path: a copy stream each way and the events that order the row chunks
    std::mutex mu_host;
    cudaStream_t copy_in = nullptr, copy_out = nullptr;
    std::vector<cudaEvent_t> host_events;
};

namespace wq {
int handle_device(wq_weights_t h) { return h->device; }
}  // namespace wq

namespace {

wq_status check_config(const wq_config* c) {
    if (!c) return fail(WQ_ERR_INVALID, "cfg is NULL");
    if (c->K <= 0 || c->N <= 0 || c->rank < 0 || c->n_outliers < 0)
        return fail(WQ_ERR_INVALID, "negative or zero size in cfg");
    if (c->mode != WQ_MODE_W4A4 && c->mode != WQ_MODE_W8A8 && c->mode != WQ_MODE_W8A8_FP8 && c->mode != WQ_MODE_W4A8)
        return fail(WQ_ERR_INVALID, "unknown mode");
    const bool eight = c->mode == WQ_MODE_W8A8 || c->mode == WQ_MODE_W8A8_FP8;
    if (c->mode == WQ_MODE_W4A8 && c->act_scale != WQ_ACT_SCALE_ROW)
        return fail(WQ_ERR_UNSUPPORTED, "WQ_MODE_W4A8 takes WQ_ACT_SCALE_ROW");
    if (eight && (c->rank != 0 || c->n_outliers != 0))
        return fail(WQ_ERR_UNSUPPORTED, "the 8-bit modes take rank 0 and no outlier channels");
    if (c->rotate != 0 && c->rotate != 1) return fail(WQ_ERR_INVALID, "rotate must be 0 or 1");
    if (c->K % 64 || c->K > 16384) return fail(WQ_ERR_UNSUPPORTED, "K must be a multiple of 64 and <= 16384");
    if (c->N % 16) return fail(WQ_ERR_UNSUPPORTED, "N must be a multiple of 16");
    if (c->rank > 64) return fail(WQ_ERR_UNSUPPORTED, "rank must be <= 64");
    if (c->n_outliers > 64 || c->n_outliers > c->K) return fail(WQ_ERR_UNSUPPORTED, "n_outliers must be <= 64 and <= K");
    if (c->act_scale != WQ_ACT_SCALE_ROW && c->act_scale != WQ_ACT_SCALE_TENSOR && c->act_scale != WQ_ACT_SCALE_STATIC)
        return fail(WQ_ERR_INVALID, "unknown act_scale");
    if (eight && c->act_scale != WQ_ACT_SCALE_ROW)
        return fail(WQ_ERR_UNSUPPORTED, "the 8-bit modes take WQ_ACT_SCALE_ROW");
    if (c->act_scale == WQ_ACT_SCALE_STATIC && !(c->act_gscale > 0.0f && std::isfinite(c->act_gscale)))
        return fail(WQ_ERR_INVALID, "WQ_ACT_SCALE_STATIC needs a finite act_gscale > 0");
    if (c->transform_order != WQ_ORDER_SMOOTH_ROTATE && c->transform_order != WQ_ORDER_ROTATE_SMOOTH)
        return fail(WQ_ERR_INVALID, "unknown transform_order");
    if (eight && c->transform_order != WQ_ORDER_SMOOTH_ROTATE)
        return fail(WQ_ERR_UNSUPPORTED, "the 8-bit modes take WQ_ORDER_SMOOTH_ROTATE");
    if (c->project != 0 && c->project != 1) return fail(WQ_ERR_INVALID, "project must be 0 or 1");
    if (c->project && (c->rank == 0 || c->mode != WQ_MODE_W4A4 || c->act_scale != WQ_ACT_SCALE_ROW ||
                       c->transform_order != WQ_ORDER_SMOOTH_ROTATE))
        return fail(WQ_ERR_UNSUPPORTED,
                    "project takes rank > 0, WQ_MODE_W4A4, WQ_ACT_SCALE_ROW and WQ_ORDER_SMOOTH_ROTATE");
    return WQ_OK;
}

void free_device(wq_weights* h) {
    cudaFree(h->d_codes);
    cudaFree(h->d_sf);
    cudaFree(h->d_sf192);
    cudaFree(h->d_bias);
    cudaFree(h->d_inv_s);
    cudaFree(h->d_inv_s_rr);
    cudaFree(h->d_omega_blk);
    cudaFree(h->d_P);
    cudaFree(h->d_Pfrag);
    cudaFree(h->d_Qt);
    cudaFree(h->d_WOt);
    cudaFree(h->d_err);
    cudaFree(h->d_colscale);
    cudaFree(h->d_amax);
    cudaFree(h->d_wexp);
    cudaFree(h->d_Vt);
    if (h->copy_in) cudaStreamDestroy(h->copy_in);
    if (h->copy_out) cudaStreamDestroy(h->copy_out);
    for (cudaEvent_t e : h->host_events) cudaEventDestroy(e);
}

template <typename T>
wq_status upload(T** dst, const void* src, size_t bytes, cudaStream_t st) {
    if (bytes == 0) return WQ_OK;
    if (cudaMalloc(reinterpret_cast<void**>(dst), bytes) != cudaSuccess)
        return fail(WQ_ERR_OOM, "cudaMalloc of " + std::to_string(bytes) + " bytes failed");
    WQ_CUDA(cudaMemcpyAsync(*dst, src, bytes, cudaMemcpyHostToDevice, st), "weight upload");
    return WQ_OK;
}

}  // namespace

// Per 32-channel half of each 64-block, channels k and k + 16 side by side (k = 0..15): the
// order in which a quantiser lane holds its channels as packed pairs.
template <typename T>
static std::vector<T> pair_order(const std::vector<T>& v) {
    std::vector<T> o(v.size());
    for (size_t h = 0; h < v.size() / 32; ++h)
        for (size_t k = 0; k < 16; ++k) {
            o[32 * h + 2 * k] = v[32 * h + k];
            o[32 * h + 2 * k + 1] = v[32 * h + k + 16];
        }
    return o;
}

extern "C" {

WQ_API const char* wq_last_error(void) { return g_last_error.c_str(); }

WQ_API wq_status wq_get_config(wq_weights_t h, wq_config* cfg) {
    if (!h || !cfg) return fail(WQ_ERR_INVALID, "NULL argument");
    *cfg = h->cfg;
    return WQ_OK;
}

WQ_API wq_status wq_prepare_weights(const wq_config* cfg, const float* W, const float* bias, const float* s,
                                    const float* L1, const float* L2, const int32_t* omega, void* stream,
                                    wq_weights_t* out) {
    g_last_error.clear();
    if (!out) return fail(WQ_ERR_INVALID, "out is NULL");
    *out = nullptr;
    wq_status st = check_config(cfg);
    if (st != WQ_OK) return st;
    if (!W) return fail(WQ_ERR_INVALID, "W is NULL");
    const int K = cfg->K, N = cfg->N, r = cfg->rank, no = cfg->n_outliers;
    // stored widths of the side operands: the extra columns of P, Q^T and W_O^T are zero, so
    // the extra U columns are exact zeros and x_O's extra columns meet zero weights
    const int rp = wq::side_width(r), nop = wq::side_width(no);
    if (r > 0 && (!L1 || !L2)) return fail(WQ_ERR_INVALID, "rank > 0 needs L1 and L2");
    if (no > 0 && !omega) return fail(WQ_ERR_INVALID, "n_outliers > 0 needs omega");
    for (int j = 0; j < no; ++j) {
        if (omega[j] < 0 || omega[j] >= K) return fail(WQ_ERR_INVALID, "omega index out of range");
        if (j > 0 && omega[j] <= omega[j - 1]) return fail(WQ_ERR_INVALID, "omega must be strictly ascending");
    }
    if (s)
        for (int k = 0; k < K; ++k)
            if (!(s[k] > 0.0f) || !std::isfinite(s[k])) return fail(WQ_ERR_INVALID, "s must be finite and > 0");

    // ---- smoothing inverse and the 16-bit low-rank factors
    std::vector<float> inv_s(s ? K : 0);
    for (int k = 0; k < (s ? K : 0); ++k) inv_s[k] = 1.0f / s[k];
    const std::vector<float> inv_s_pairs = pair_order(inv_s);
    // rotation first (QuantWAMs Eq. (1)): smoothing applies in the rotated basis
    const bool after = cfg->transform_order == WQ_ORDER_ROTATE_SMOOTH && cfg->rotate;
    std::vector<uint16_t> P(static_cast<size_t>(K) * rp, 0), Qt(static_cast<size_t>(N) * rp, 0);
    if (!after) {
        for (int k = 0; k < K; ++k)
            for (int j = 0; j < r; ++j) {
                float l = L1[static_cast<size_t>(k) * r + j];
                if (s) l = l * inv_s[k];
                P[static_cast<size_t>(k) * rp + j] = bf16_bits(l);
            }
    } else {
        // P = H diag(1/s) L1, fp64, one rounding to bf16
        std::vector<double> col(K);
        for (int j = 0; j < r; ++j) {
            for (int k = 0; k < K; ++k)
                col[k] = static_cast<double>(L1[static_cast<size_t>(k) * r + j]) * (s ? static_cast<double>(inv_s[k]) : 1.0);
            for (int b = 0; b < K / 64; ++b) fwht64_f64(col.data() + 64 * b, 1);
            for (int k = 0; k < K; ++k) P[static_cast<size_t>(k) * rp + j] = bf16_bits_from_f64(col[k]);
        }
    }
    // P as the B operand of mma.sync.m16n8k16 (k16 x n8 tiles): for 64-block kb, n-tile nt,
    // lane (g = lane / 4, c = lane % 4) and k16 step f, the lane's two registers hold
    // {P[k][j], P[k+1][j]} and {P[k+8][j], P[k+9][j]} with k = 64 kb + 16 f + 2 c, j = 8 nt + g.
    std::vector<uint32_t> Pfrag(static_cast<size_t>(K) * rp / 2);
    if (r > 0) {
        const int NT = rp / 8;
        for (int kb = 0; kb < K / 64; ++kb)
            for (int nt = 0; nt < NT; ++nt)
                for (int lane = 0; lane < 32; ++lane)
                    for (int f = 0; f < 4; ++f) {
                        const int g = lane / 4, c = lane % 4, j = 8 * nt + g, k = 64 * kb + 16 * f + 2 * c;
                        auto at = [&](int kk) { return static_cast<uint32_t>(P[static_cast<size_t>(kk) * rp + j]); };
                        const size_t o = ((static_cast<size_t>(kb) * NT + nt) * 32 + lane) * 8 + 2 * f;
                        Pfrag[o] = at(k) | (at(k + 1) << 16);
                        Pfrag[o + 1] = at(k + 8) | (at(k + 9) << 16);
                    }
    }
    std::vector<float> Pf(static_cast<size_t>(K) * r), Qf(static_cast<size_t>(r) * N);
    for (int k = 0; k < K; ++k)
        for (int j = 0; j < r; ++j)
            Pf[static_cast<size_t>(k) * r + j] = __bfloat162float(__ushort_as_bfloat16(P[static_cast<size_t>(k) * rp + j]));
    for (int j = 0; j < r; ++j)
        for (int n = 0; n < N; ++n) {
            const uint16_t b = bf16_bits(L2[static_cast<size_t>(j) * N + n]);
            Qt[static_cast<size_t>(n) * rp + j] = b;
            Qf[static_cast<size_t>(j) * N + n] = __bfloat162float(__ushort_as_bfloat16(b));
        }

    // ---- fold: R' = FWHT_64( diag(s) (W - P Q) ) along K, fp64, rounded once to fp32
    std::vector<float> Rp(static_cast<size_t>(K) * N);
    parallel_for(static_cast<size_t>(N), [&](size_t n) {
        std::vector<double> col(K);
        for (int k = 0; k < K; ++k) {
            double lr = 0.0;
            for (int j = 0; j < r; ++j)
                lr += static_cast<double>(Pf[static_cast<size_t>(k) * r + j]) *
                      static_cast<double>(Qf[static_cast<size_t>(j) * N + n]);
            const double t = static_cast<double>(W[static_cast<size_t>(k) * N + n]) - lr;
            col[k] = (s && !after) ? static_cast<double>(s[k]) * t : t;
        }
        if (cfg->rotate)
            for (int b = 0; b < K / 64; ++b) fwht64_f64(col.data() + 64 * b, 1);
        if (s && after)
            for (int k = 0; k < K; ++k) col[k] = static_cast<double>(s[k]) * col[k];
        for (int k = 0; k < K; ++k) Rp[static_cast<size_t>(k) * N + n] = static_cast<float>(col[k]);
    });

    // ---- the fp16 outlier rows of the rotated basis
    std::vector<uint16_t> WOt(static_cast<size_t>(N) * nop, 0);
    // per 64-block of K: which channels are kept (bit mask) and the x_O index of the first one
    std::vector<uint32_t> omega_blk(no ? static_cast<size_t>(K / 64) * 4 : 0, 0u);
    for (int j = no - 1; j >= 0; --j) {
        const int b = omega[j] / 64, e = omega[j] % 64;
        omega_blk[4 * b + e / 32] |= 1u << (e % 32);
        omega_blk[4 * b + 2] = static_cast<uint32_t>(j);
    }
    for (int j = 0; j < no; ++j) {
        for (int n = 0; n < N; ++n) {
            float& v = Rp[static_cast<size_t>(omega[j]) * N + n];
            WOt[static_cast<size_t>(n) * nop + j] = f16_bits(v);
            v = 0.0f;
        }
    }

    if (cfg->mode == WQ_MODE_W8A8 || cfg->mode == WQ_MODE_W8A8_FP8) {
        // ---- symmetric 8-bit per output column, K-major: int8 values kept as exact bf16 integers,
        // or e4m3 bytes (scale amax / 448, code e4m3_rn_satfinite(RN(v / scale)))
        const bool f8 = cfg->mode == WQ_MODE_W8A8_FP8;
        std::vector<uint16_t> q8(f8 ? 0 : static_cast<size_t>(N) * K);
        std::vector<uint8_t> e8(f8 ? static_cast<size_t>(N) * K : 0);
        std::vector<float> wsc(N);
        parallel_for(static_cast<size_t>(N), [&](size_t n) {
            float am = 0.0f;
            for (int k = 0; k < K; ++k) am = std::max(am, std::fabs(Rp[static_cast<size_t>(k) * N + n]));
            const float sc = am / (f8 ? 448.0f : 127.0f);
            wsc[n] = sc;
            for (int k = 0; k < K; ++k) {
                if (f8) {
                    uint8_t c = 0;
                    if (sc != 0.0f)
                        c = static_cast<uint8_t>(__nv_cvt_float_to_fp8(Rp[static_cast<size_t>(k) * N + n] / sc,
                                                                       __NV_SATFINITE, __NV_E4M3));
                    e8[n * K + k] = c;
                    continue;
                }
                float r = 0.0f;
                if (sc != 0.0f) r = std::nearbyint(Rp[static_cast<size_t>(k) * N + n] / sc);
                r = std::min(127.0f, std::max(-127.0f, r));
                q8[n * K + k] = bf16_bits(r);
            }
        });
        wq_weights* h = new (std::nothrow) wq_weights();
        if (!h) return fail(WQ_ERR_OOM, "host allocation failed");
        h->cfg = *cfg;
        h->gW = 1.0f;
        cudaStream_t cs = static_cast<cudaStream_t>(stream);
        auto bail = [&](wq_status e) { free_device(h); delete h; return e; };
        if (cudaGetDevice(&h->device) != cudaSuccess) return bail(fail(WQ_ERR_CUDA, "cudaGetDevice failed"));
        cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
        std::vector<float> bias_f(N, 0.0f);
        if (bias) std::copy(bias, bias + N, bias_f.begin());
        if (f8) {
            if ((st = upload(&h->d_codes, e8.data(), e8.size(), cs)) != WQ_OK) return bail(st);
        } else if ((st = upload(&h->d_codes, q8.data(), q8.size() * 2, cs)) != WQ_OK) {
            return bail(st);
        }
        if ((st = upload(&h->d_colscale, wsc.data(), N * 4, cs)) != WQ_OK) return bail(st);
        if (bias && (st = upload(&h->d_bias, bias_f.data(), N * 4, cs)) != WQ_OK) return bail(st);
        if (s && (st = upload(&h->d_inv_s, inv_s_pairs.data(), K * 4, cs)) != WQ_OK) return bail(st);
        if (cudaMalloc(&h->d_err, sizeof(int)) != cudaSuccess) return bail(fail(WQ_ERR_OOM, "cudaMalloc failed"));
        if (cudaMemsetAsync(h->d_err, 0, sizeof(int), cs) != cudaSuccess) return bail(fail(WQ_ERR_CUDA, "memset"));
        if (cudaStreamSynchronize(cs) != cudaSuccess) return bail(fail(WQ_ERR_CUDA, "upload synchronise failed"));
        const char* why = "";
        const bool okm = f8 ? wq::encode_tmap_2d(&h->tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->d_codes, K, N, K, 128, 128,
                                                 CU_TENSOR_MAP_SWIZZLE_128B, &why)
                            : wq::encode_tmap_2d(&h->tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->d_codes, K, N, 2ull * K,
                                                 64, 128, CU_TENSOR_MAP_SWIZZLE_128B, &why);
        if (!okm) return bail(fail(WQ_ERR_CUDA, why));
        *out = h;
        return WQ_OK;
    }

    // ---- NVFP4 with one fp32 scale for the tensor; column n quantised along K
    float amax = 0.0f;
    for (float v : Rp) amax = std::max(amax, std::fabs(v));
    const float gW = amax / 2688.0f;
    const size_t n_pad = align_up(static_cast<size_t>(N), wq::kBlockM);
    std::vector<uint8_t> codes(static_cast<size_t>(N) * K / 2);
    std::vector<uint8_t> sf_mma(n_pad / wq::kBlockM * (K / 64) * wq::kSfAtom, 0);
    parallel_for(static_cast<size_t>(N), [&](size_t n) {
        for (int b = 0; b < K / 16; ++b) {
            float v[16], bmax = 0.0f;
            for (int i = 0; i < 16; ++i) {
                v[i] = Rp[static_cast<size_t>(16 * b + i) * N + n];
                bmax = std::max(bmax, std::fabs(v[i]));
            }
            uint32_t sc = 0;
            if (gW != 0.0f) {
                const float t = bmax / 6.0f;
                sc = static_cast<uint32_t>(__nv_cvt_float_to_fp8(t / gW, __NV_SATFINITE, __NV_E4M3));
            }
            const float d = e4m3_value(sc) * gW;
            for (int i = 0; i < 16; i += 2) {
                uint32_t c0 = 0, c1 = 0;
                if (d != 0.0f) {
                    c0 = __nv_cvt_float_to_fp4(v[i] / d, __NV_E2M1, cudaRoundNearest) & 15u;
                    c1 = __nv_cvt_float_to_fp4(v[i + 1] / d, __NV_E2M1, cudaRoundNearest) & 15u;
                }
                codes[n * (K / 2) + 8 * b + i / 2] = static_cast<uint8_t>(c0 | (c1 << 4));
            }
            const size_t row = n, kb = static_cast<size_t>(b) / 4;
            const size_t off = ((row / wq::kBlockM) * (K / 64) + kb) * wq::kSfAtom + (row % 32) * 16 +
                               ((row % wq::kBlockM) / 32) * 4 + (b % 4);
            sf_mma[off] = static_cast<uint8_t>(sc);
        }
    });

    // ---- device residency
    wq_weights* h = new (std::nothrow) wq_weights();
    if (!h) return fail(WQ_ERR_OOM, "host allocation failed");
    h->cfg = *cfg;
    h->gW = gW;
    h->r_pad = rp;
    h->no_pad = nop;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    auto bail = [&](wq_status e) { free_device(h); delete h; return e; };
    if (cudaGetDevice(&h->device) != cudaSuccess) return bail(fail(WQ_ERR_CUDA, "cudaGetDevice failed"));
    cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
    std::vector<float> bias_f(N, 0.0f);
    if (bias) std::copy(bias, bias + N, bias_f.begin());
    if ((st = upload(&h->d_codes, codes.data(), codes.size(), cs)) != WQ_OK) return bail(st);
    if ((st = upload(&h->d_sf, sf_mma.data(), sf_mma.size(), cs)) != WQ_OK) return bail(st);
    // the same scales in 192-row tile layout: tile t's rows 0..127 in atom block 2 t, rows 128..191
    // in the first half of atom block 2 t + 1 (the rest zero)
    const size_t nt192 = (static_cast<size_t>(N) + 191) / 192, nkb = static_cast<size_t>(K / 64);
    std::vector<uint8_t> sf192(nt192 * 2 * nkb * wq::kSfAtom, 0);
    for (size_t n = 0; n < static_cast<size_t>(N); ++n) {
        const size_t t = n / 192, m = (n % 192) % 128, z = 2 * t + (n % 192) / 128;
        for (size_t kb = 0; kb < nkb; ++kb)
            for (size_t j = 0; j < 4; ++j) {
                const size_t src = ((n / wq::kBlockM) * nkb + kb) * wq::kSfAtom + (n % 32) * 16 + ((n % wq::kBlockM) / 32) * 4 + j;
                const size_t dst = (z * nkb + kb) * wq::kSfAtom + (m % 32) * 16 + (m / 32) * 4 + j;
                sf192[dst] = sf_mma[src];
            }
    }
    if ((st = upload(&h->d_sf192, sf192.data(), sf192.size(), cs)) != WQ_OK) return bail(st);
    if (bias && (st = upload(&h->d_bias, bias_f.data(), N * 4, cs)) != WQ_OK) return bail(st);
    if (s && (st = upload(&h->d_inv_s, inv_s_pairs.data(), K * 4, cs)) != WQ_OK) return bail(st);
    std::vector<float> inv_s_rr(s ? K : 0);
    for (int k = 0; k < (s ? K : 0); ++k) inv_s_rr[k] = inv_s[(k / 64) * 64 + (k % 64) / 2 + 32 * (k % 2)];
    if (s && (st = upload(&h->d_inv_s_rr, inv_s_rr.data(), K * 4, cs)) != WQ_OK) return bail(st);
    if (no && (st = upload(&h->d_omega_blk, omega_blk.data(), omega_blk.size() * 4, cs)) != WQ_OK) return bail(st);
    if (r && (st = upload(&h->d_P, P.data(), P.size() * 2, cs)) != WQ_OK) return bail(st);
    if (r && (st = upload(&h->d_Pfrag, Pfrag.data(), Pfrag.size() * 4, cs)) != WQ_OK) return bail(st);
    if (r && (st = upload(&h->d_Qt, Qt.data(), Qt.size() * 2, cs)) != WQ_OK) return bail(st);
    if (no && (st = upload(&h->d_WOt, WOt.data(), WOt.size() * 2, cs)) != WQ_OK) return bail(st);
    if (cudaMalloc(&h->d_err, sizeof(int)) != cudaSuccess) return bail(fail(WQ_ERR_OOM, "cudaMalloc failed"));
    if (cudaMemsetAsync(h->d_err, 0, sizeof(int), cs) != cudaSuccess) return bail(fail(WQ_ERR_CUDA, "memset"));
    if (cfg->act_scale == WQ_ACT_SCALE_TENSOR &&
        cudaMalloc(reinterpret_cast<void**>(&h->d_amax), 16) != cudaSuccess)
        return bail(fail(WQ_ERR_OOM, "cudaMalloc failed"));
    if (cudaStreamSynchronize(cs) != cudaSuccess) return bail(fail(WQ_ERR_CUDA, "upload synchronise failed"));

    const char* why = "";
    if (!wq::encode_tmap_2d(&h->tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->d_codes, K / 2, N, K / 2, 128, 128,
                            CU_TENSOR_MAP_SWIZZLE_128B, &why) ||
        !wq::encode_scale_tmap(&h->tmSFB, h->d_sf, N, K, 2, &why) ||
        !wq::encode_tmap_2d(&h->tmB96, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->d_codes, K / 2, N, K / 2, 128, 96,
                            CU_TENSOR_MAP_SWIZZLE_128B, &why) ||
        !wq::encode_scale_tmap_blocks(&h->tmSFB192, h->d_sf192, static_cast<int>(2 * nt192), K, 2, &why) ||
        !wq::encode_tmap_2d(&h->tmBconv, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->d_codes, K / 2, N, K / 2, 64, 128,
                            CU_TENSOR_MAP_SWIZZLE_64B, &why))
        return bail(fail(WQ_ERR_CUDA, why));
    if (r && (!wq::encode_tmap_2d(&h->tmQ, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->d_Qt, rp, N, 2 * rp, rp, 128,
                                  swizzle_for_row_bytes(2 * rp), &why) ||
              !wq::encode_tmap_2d(&h->tmQ96, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->d_Qt, rp, N, 2 * rp, rp, 96,
                                  swizzle_for_row_bytes(2 * rp), &why)))
        return bail(fail(WQ_ERR_CUDA, why));
    if (no && (!wq::encode_tmap_2d(&h->tmWO, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, h->d_WOt, nop, N, 2 * nop, nop, 128,
                                   swizzle_for_row_bytes(2 * nop), &why) ||
               !wq::encode_tmap_2d(&h->tmWO96, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, h->d_WOt, nop, N, 2 * nop, nop, 96,
                                   swizzle_for_row_bytes(2 * nop), &why)))
        return bail(fail(WQ_ERR_CUDA, why));
    if (cfg->mode == WQ_MODE_W4A8) {
        // A8 steps multiply the NVFP4 weights on the 16-bit tensor path: each value dec(code) dec(scale)
        // has at most 6 significant bits and lies in [2^-10, 2688], so bf16 holds it exactly (gW stays
        // in the epilogue)
        std::vector<uint16_t> wexp(static_cast<size_t>(N) * K);
        parallel_for(static_cast<size_t>(N), [&](size_t n) {
            for (int k = 0; k < K; ++k) {
                const uint32_t byte = codes[n * (K / 2) + k / 2];
                const uint32_t c = (k & 1) ? (byte >> 4) : (byte & 15u);
                const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
                const size_t off = ((n / wq::kBlockM) * (K / 64) + k / 64) * wq::kSfAtom + (n % 32) * 16 +
                                   ((n % wq::kBlockM) / 32) * 4 + (k % 64) / 16;
                const float v = ((c & 8u) ? -mag[c & 7u] : mag[c & 7u]) * e4m3_value(sf_mma[off]);
                wexp[n * K + k] = bf16_bits(v);
            }
        });
        if ((st = upload(&h->d_wexp, wexp.data(), wexp.size() * 2, cs)) != WQ_OK) return bail(st);
        if (cudaStreamSynchronize(cs) != cudaSuccess) return bail(fail(WQ_ERR_CUDA, "upload synchronise failed"));
        if (!wq::encode_tmap_2d(&h->tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, h->d_wexp, K, N, 2ull * K, 64, 128,
                                CU_TENSOR_MAP_SWIZZLE_128B, &why))
            return bail(fail(WQ_ERR_CUDA, why));
    }
    if (cfg->project) {
        // Vt[j] = FWHT_64(L1[:, j]) / ||L1[:, j]||^2, fp64, one rounding to bf16
        std::vector<uint16_t> Vt(static_cast<size_t>(r) * K);
        std::vector<double> col(K);
        for (int j = 0; j < r; ++j) {
            double nrm = 0.0;
            for (int k = 0; k < K; ++k) {
                col[k] = static_cast<double>(L1[static_cast<size_t>(k) * r + j]);
                nrm += col[k] * col[k];
            }
            if (cfg->rotate)
                for (int b = 0; b < K / 64; ++b) fwht64_f64(col.data() + 64 * b, 1);
            for (int k = 0; k < K; ++k)
                Vt[static_cast<size_t>(j) * K + k] = bf16_bits_from_f64(nrm > 0.0 ? col[k] / nrm : 0.0);
        }
        if ((st = upload(&h->d_Vt, Vt.data(), Vt.size() * 2, cs)) != WQ_OK) return bail(st);
        if (cudaStreamSynchronize(cs) != cudaSuccess) return bail(fail(WQ_ERR_CUDA, "upload synchronise failed"));
    }
    *out = h;
    return WQ_OK;
}

// 8-bit codes [M, K] (bf16-held int8: 2 bytes, e4m3: 1 byte) and the row scales
static size_t w8_code_bytes(wq_weights_t h, int M) {
    return static_cast<size_t>(M) * h->cfg.K * (h->cfg.mode == WQ_MODE_W8A8_FP8 ? 1 : 2);
}
static size_t w8_workspace_bytes(wq_weights_t h, int M) {
    return align_up(w8_code_bytes(h, M), 1024) + align_up(static_cast<size_t>(M) * 4, 1024);
}

// W4A8: the e4m3 activation values as bf16 [M, K] in place of the fp4 codes (4 x their bytes: the
// fp4-code region of a 4K-wide carve), the row scales, U, x_O and the batch-maximum word
static wq::ActWorkspace carve_w4a8(void* base, int M, int K, int r, int no) {
    return wq::carve_workspace(base, M, 4 * K, r, no);
}

WQ_API size_t wq_workspace_bytes(wq_weights_t h, int M) {
    if (!h || M < 0) return 0;
    if (h->cfg.mode == WQ_MODE_W4A8) return carve_w4a8(nullptr, M, h->cfg.K, h->r_pad, h->no_pad).bytes;
    if (h->cfg.mode != WQ_MODE_W4A4) return w8_workspace_bytes(h, M);
    return wq::carve_workspace(nullptr, M, h->cfg.K, h->r_pad, h->no_pad).bytes;
}

WQ_API wq_status wq_side_strides(wq_weights_t h, int* u_ld, int* xo_ld) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (u_ld) *u_ld = h->r_pad;
    if (xo_ld) *xo_ld = h->no_pad;
    return WQ_OK;
}

WQ_API wq_status wq_set_tuning(const char* name, int value) {
    const int k = wq::knob_index(name);
    if (k < 0) return fail(WQ_ERR_INVALID, std::string("unknown tuning knob ") + (name ? name : "(null)"));
    wq::tune(static_cast<wq::TuneKnob>(k));             // the environment is read first, once
    wq::g_knob[k].store(value, std::memory_order_relaxed);
    return WQ_OK;
}

WQ_API int wq_get_tuning(const char* name) {
    const int k = wq::knob_index(name);
    if (k < 0) return fail(WQ_ERR_INVALID, std::string("unknown tuning knob ") + (name ? name : "(null)"));
    return wq::tune(static_cast<wq::TuneKnob>(k));
}

WQ_API size_t wq_host_workspace_bytes(wq_weights_t h, int M) {
    if (!h || M < 0) return 0;
    return wq_workspace_bytes(h, M) + align_up(static_cast<size_t>(M) * h->cfg.K * 2, 1024) +
           align_up(static_cast<size_t>(M) * h->cfg.N * 2, 1024);
}

// Launching entry points run on the handle's device only: its weights, error flag and scratch
// live there.
static wq_status check_device(wq_weights_t h) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return fail(WQ_ERR_CUDA, "cudaGetDevice failed");
    if (dev != h->device)
        return fail(WQ_ERR_INVALID, "the current device (" + std::to_string(dev) + ") is not the handle's device (" +
                                        std::to_string(h->device) + ")");
    return WQ_OK;
}

// x as [M, K] bf16 in 16-row x 64-channel boxes (re-encoded when x or M changes).  The map is
// copied out under the lock: the launch passes it by value, so a concurrent call on the same
// handle that re-encodes the cached map cannot change what this launch reads.
static wq_status x_map(wq_weights_t h, const void* x, int M, CUtensorMap* out) {
    std::lock_guard<std::mutex> lk(h->mu_x);
    if (h->key_x != x || h->key_xM != M) {
        const char* why = "";
        if (!wq::encode_tmap_2d(&h->tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, x, h->cfg.K, M, 2ull * h->cfg.K, 64, 16,
                                CU_TENSOR_MAP_SWIZZLE_128B, &why)) {
            h->key_x = nullptr;
            return fail(WQ_ERR_CUDA, why);
        }
        h->key_x = x;
        h->key_xM = M;
    }
    *out = h->tmX;
    return WQ_OK;
}

static wq_status run_quant(wq_weights_t h, const void* x, int M, int layout, uint8_t* codes, uint8_t* sf, float* g,
                           uint16_t* xo, uint16_t* u, unsigned int* amax, cudaStream_t st) {
    wq::QuantArgs qa{};
    CUtensorMap tmx;
    {
        const wq_status s = x_map(h, x, M, &tmx);
        if (s != WQ_OK) return s;
        qa.tmX = &tmx;
    }
    qa.act_scale = h->cfg.act_scale;
    qa.static_g = h->cfg.act_gscale;
    if (qa.act_scale == WQ_ACT_SCALE_TENSOR) {
        qa.amax_bits = amax;
        WQ_CUDA(cudaMemsetAsync(amax, 0, sizeof(unsigned int), st), "batch maximum reset");
    }
    qa.pfrag = h->d_Pfrag;
    qa.err = h->d_err;
    qa.x = x;
    qa.M = M;
    qa.K = h->cfg.K;
    qa.inv_s = h->d_inv_s;
    qa.inv_s_rr = h->d_inv_s_rr;
    qa.rotate = h->cfg.rotate | (h->cfg.rotate && h->cfg.transform_order == WQ_ORDER_ROTATE_SMOOTH ? 2 : 0);
    qa.omega_blk = h->d_omega_blk;
    qa.n_out = xo ? h->cfg.n_outliers : 0;
    qa.xo_ld = h->no_pad;
    qa.xo = xo;
    qa.P = h->d_P;
    qa.r = u ? h->r_pad : 0;
    qa.u = u;
    qa.codes = codes;
    qa.sf = sf;
    qa.sf_layout = layout;
    qa.g = g;
    qa.num_sms = h->num_sms;
    qa.int8 = h->cfg.mode != WQ_MODE_W4A4;
    qa.fp8 = h->cfg.mode == WQ_MODE_W8A8_FP8 || h->cfg.mode == WQ_MODE_W4A8;
    qa.fp8_bf16 = h->cfg.mode == WQ_MODE_W4A8;
    if (h->cfg.project) {
        if (!u) return fail(WQ_ERR_INVALID, "project: the U buffer is required (u = x P feeds the projection)");
        qa.vt = h->d_Vt;
        qa.r_real = h->cfg.rank;
    }
    const cudaError_t e = wq::launch_quantize_act(qa, st);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantiser launch");
    return WQ_OK;
}

WQ_API wq_status wq_quantize_activations(wq_weights_t h, const void* x, int M, int scale_layout, uint8_t* codes,
                                         uint8_t* scales, float* gscale, void* x_omega, void* u, void* stream) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    if (M == 0) return WQ_OK;
    if (!x || !codes || (!scales && h->cfg.mode == WQ_MODE_W4A4) || !gscale) return fail(WQ_ERR_INVALID, "NULL buffer");
    if (h->cfg.mode != WQ_MODE_W4A4 && h->cfg.mode != WQ_MODE_W4A8)
        return fail(WQ_ERR_INVALID, "W8A8 handle: use wq_quantize_activations_w8a8");
    if (h->cfg.n_outliers > 0 && !x_omega)
        return fail(WQ_ERR_INVALID, "x_omega is required when n_outliers > 0 (the kept channels are zeroed)");
    if (scale_layout != WQ_SCALE_LAYOUT_ROWMAJOR && scale_layout != WQ_SCALE_LAYOUT_MMA)
        return fail(WQ_ERR_INVALID, "bad scale_layout");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(scales)) & 15)
        return fail(WQ_ERR_INVALID, "device buffers must be 16-byte aligned");
    if (const wq_status d = check_device(h)) return d;
    return run_quant(h, x, M, scale_layout, codes, scales, gscale,
                     h->cfg.n_outliers ? static_cast<uint16_t*>(x_omega) : nullptr,
                     h->cfg.rank ? static_cast<uint16_t*>(u) : nullptr, h->d_amax, static_cast<cudaStream_t>(stream));
}

static wq_status run_gemm(wq_weights_t h, const uint8_t* codes, const uint8_t* sf, const float* g,
                          const uint16_t* u, const uint16_t* xo, int M, void* y, cudaStream_t st,
                          const wq::ChainArgs* chain = nullptr) {
    const int K = h->cfg.K, N = h->cfg.N, r = h->r_pad, no = h->no_pad, no_real = h->cfg.n_outliers;
    std::lock_guard<std::mutex> lk(h->mu);
    if (h->key_codes != codes || h->key_u != u || h->key_xo != xo || h->key_y != y || h->key_sf != sf ||
        h->key_M != M) {
        const char* why = "";
        const bool w8 = h->cfg.mode == WQ_MODE_W8A8 || h->cfg.mode == WQ_MODE_W4A8, f8 = h->cfg.mode == WQ_MODE_W8A8_FP8;
        bool ok = (w8 ? wq::encode_tmap_2d(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, codes, K, M, 2ull * K, 64, 128,
                                           CU_TENSOR_MAP_SWIZZLE_128B, &why)
                      : f8 ? wq::encode_tmap_2d(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K, M, K, 128, 128,
                                                CU_TENSOR_MAP_SWIZZLE_128B, &why)
                           : wq::encode_tmap_2d(&h->tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, codes, K / 2, M, K / 2, 128, 128,
                                                CU_TENSOR_MAP_SWIZZLE_128B, &why)) &&
                  wq::encode_tmap_2d(&h->tmY, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, N, M, 2ull * N, 64, 32,
                                     CU_TENSOR_MAP_SWIZZLE_128B, &why);
        if (ok && !w8 && !f8)
            ok = wq::encode_scale_tmap(&h->tmSFA, sf, M, K, 1, &why) &&
                 wq::encode_tmap_2d(&h->tmY32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, y, N, M, 2ull * N, 32, 32,
                                    CU_TENSOR_MAP_SWIZZLE_NONE, &why);
        if (ok && r)
            ok = wq::encode_tmap_2d(&h->tmU, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, u, r, M, 2 * r, r, 128,
                                    swizzle_for_row_bytes(2 * r), &why);
        // x_O's columns beyond the real count are read as zeros (outside the map's extent)
        if (ok && no)
            ok = wq::encode_tmap_2d(&h->tmXO, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, xo, no_real, M, 2 * no, no, 128,
                                    swizzle_for_row_bytes(2 * no), &why);
        if (!ok) {
            h->key_codes = nullptr;
            return fail(WQ_ERR_CUDA, why);
        }
        h->key_codes = codes;
        h->key_u = u;
        h->key_xo = xo;
        h->key_y = y;
        h->key_sf = sf;
        h->key_M = M;
    }
    wq::GemmArgs ga{};
    ga.M = M; ga.N = N; ga.K = K; ga.r = r; ga.n_out = no;
    ga.tmA = &h->tmA; ga.tmB = &h->tmB; ga.tmU = &h->tmU; ga.tmQ = &h->tmQ;
    ga.tmXO = &h->tmXO; ga.tmWO = &h->tmWO; ga.tmY = &h->tmY;
    ga.tmSFA = &h->tmSFA; ga.tmSFB = &h->tmSFB;
    ga.tmB96 = &h->tmB96; ga.tmQ96 = &h->tmQ96; ga.tmWO96 = &h->tmWO96; ga.tmSFB192 = &h->tmSFB192;
    ga.tmY32 = &h->tmY32;
    ga.sfa = sf; ga.sfb = h->d_sf; ga.gA = g; ga.gW = h->gW; ga.bias = h->d_bias;
    ga.err = h->d_err; ga.num_sms = h->num_sms;
    ga.y = y;
    ga.w8 = h->cfg.mode != WQ_MODE_W4A4;
    ga.fp8 = h->cfg.mode == WQ_MODE_W8A8_FP8;
    ga.colscale = h->d_colscale;
    ga.force_split = wq::tune(wq::kTuneGemmSplit);     // 0: choose (tests and tuning pin it)
    ga.chain = chain;
    if (chain) ga.force_split = 0;
    const cudaError_t e = wq::launch_gemm(ga, st);
    if (e != cudaSuccess) return cuda_fail(e, "GEMM launch");
    return WQ_OK;
}

namespace {
bool use_fused(wq_weights_t h, int M, int& nb, int& cs) {
    return h->cfg.mode == WQ_MODE_W4A4 && h->cfg.act_scale == WQ_ACT_SCALE_ROW && !h->cfg.project &&
           h->cfg.transform_order == WQ_ORDER_SMOOTH_ROTATE && wq::tune(wq::kTuneFused) == 1 &&
           wq::fused_plan(M, h->cfg.K, h->cfg.N, h->r_pad, h->no_pad, nb, cs);
}
}  // namespace

WQ_API int wq_quant_schedule(wq_weights_t h, int M) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    // batch-wide tensor scales take the stream kernel (its two-launch and one-pass forms)
    if (h->cfg.act_scale != WQ_ACT_SCALE_ROW || h->cfg.project) return WQ_QUANT_STREAM;
    if (!wq::quant_stream_schedule(M, h->num_sms)) return WQ_QUANT_CLUSTER;
    wq::QuantArgs qa{};
    qa.K = h->cfg.K;
    qa.r = h->r_pad;
    qa.int8 = h->cfg.mode != WQ_MODE_W4A4;
    qa.inv_s = h->d_inv_s;
    qa.inv_s_rr = h->d_inv_s_rr;
    return wq::tune(wq::kTuneQuantSchedule) != 1 && wq::quant_resident_eligible(qa) ? WQ_QUANT_RESIDENT
                                                                                    : WQ_QUANT_STREAM;
}

WQ_API int wq_gemm_schedule(wq_weights_t h, int M) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    wq::GemmArgs ga{};
    ga.M = M > 0 ? M : 1; ga.N = h->cfg.N; ga.K = h->cfg.K; ga.r = h->r_pad; ga.n_out = h->no_pad;
    ga.w8 = h->cfg.mode != WQ_MODE_W4A4;
    ga.fp8 = h->cfg.mode == WQ_MODE_W8A8_FP8;
    ga.num_sms = h->num_sms;
    ga.force_split = wq::tune(wq::kTuneGemmSplit);
    const int s = wq::gemm_schedule(ga);
    if (s < 0) return fail(WQ_ERR_CUDA, "GEMM schedule query failed");
    return s;
}

WQ_API int wq_forward_path(wq_weights_t h, int M) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    int nb = 0, cs = 0;
    return M > 0 && use_fused(h, M, nb, cs) ? WQ_PATH_FUSED : WQ_PATH_TWO_KERNEL;
}

WQ_API wq_status wq_linear_forward(wq_weights_t h, const void* x, int M, void* y, void* workspace,
                                   size_t workspace_bytes, void* stream) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    if (M == 0) return WQ_OK;
    if (!x || !y || !workspace) return fail(WQ_ERR_INVALID, "NULL buffer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15)
        return fail(WQ_ERR_INVALID, "x and y must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(WQ_ERR_INVALID, "workspace must be 256-byte aligned");
    if (h->cfg.mode != WQ_MODE_W4A4 && h->cfg.mode != WQ_MODE_W4A8)
        return fail(WQ_ERR_INVALID, "W8A8 handle: use wq_linear_forward_w8a8");
    if (const wq_status d = check_device(h)) return d;
    const int K = h->cfg.K, r = h->r_pad, no = h->no_pad;
    if (h->cfg.mode == WQ_MODE_W4A8) {
        // an A8-protected step: e4m3 activations (as exact bf16) times the bf16-held NVFP4 weights
        const wq::ActWorkspace w8 = carve_w4a8(workspace, M, K, r, no);
        if (workspace_bytes < w8.bytes) return fail(WQ_ERR_INVALID, "workspace too small");
        cudaStream_t st8 = static_cast<cudaStream_t>(stream);
        wq_status s8 = run_quant(h, x, M, WQ_SCALE_LAYOUT_ROWMAJOR, w8.codes, nullptr, w8.g, no ? w8.xo : nullptr,
                                 r ? w8.u : nullptr, w8.amax, st8);
        if (s8 != WQ_OK) return s8;
        return run_gemm(h, w8.codes, nullptr, w8.g, w8.u, w8.xo, M, y, st8);
    }
    const wq::ActWorkspace ws = wq::carve_workspace(workspace, M, K, r, no);
    if (workspace_bytes < ws.bytes) return fail(WQ_ERR_INVALID, "workspace too small");
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    // WQ_FUSED=1: small batches run quantiser and GEMM fused in one cluster kernel.  Opt-in:
    // on the measured batch-1 layers the two-kernel pair overlapped by programmatic dependent
    // launch is faster (the fused kernel's one-CTA-per-SM footprint also keeps the next
    // layer's quantiser from starting early).
    int nb = 0, cs = 0;
    if (use_fused(h, M, nb, cs)) {
        CUtensorMap tmx;
        wq_status s = x_map(h, x, M, &tmx);
        if (s != WQ_OK) return s;
        wq::FusedArgs fa{};
        fa.M = M; fa.K = K; fa.N = h->cfg.N; fa.r = r; fa.n_out = no; fa.nb = nb; fa.cs = cs;
        fa.tmX = &tmx; fa.tmB = nb == 4 ? &h->tmB : &h->tmBconv; fa.tmQ = &h->tmQ; fa.tmWO = &h->tmWO;
        fa.inv_s = h->d_inv_s; fa.rotate = h->cfg.rotate; fa.omega_blk = h->d_omega_blk; fa.pfrag = h->d_Pfrag;
        fa.sfb = h->d_sf; fa.gW = h->gW; fa.bias = h->d_bias; fa.y = y; fa.err = h->d_err;
        const cudaError_t e = wq::launch_fused(fa, st);
        if (e != cudaSuccess) return cuda_fail(e, "fused forward launch");
        return WQ_OK;
    }
    wq_status s = run_quant(h, x, M, WQ_SCALE_LAYOUT_MMA, ws.codes, ws.sf, ws.g, no ? ws.xo : nullptr,
                            r ? ws.u : nullptr, ws.amax, st);
    if (s != WQ_OK) return s;
    return run_gemm(h, ws.codes, ws.sf, ws.g, ws.u, ws.xo, M, y, st);
}

WQ_API wq_status wq_linear_forward_chain(wq_weights_t h, wq_weights_t next, const void* x, int M, uint8_t* codes,
                                         uint8_t* scales_mma, float* gscale, void* x_omega, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    if (!h || !next) return fail(WQ_ERR_INVALID, "NULL handle");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    if (M == 0) return WQ_OK;
    if (h->cfg.mode != WQ_MODE_W4A4 || next->cfg.mode != WQ_MODE_W4A4 || h->conv_cin || next->conv_cin)
        return fail(WQ_ERR_INVALID, "both handles must be 4-bit linear layers");
    if (next->cfg.K != h->cfg.N) return fail(WQ_ERR_INVALID, "next layer's K differs from this layer's N");
    if (next->cfg.act_scale != WQ_ACT_SCALE_STATIC)
        return fail(WQ_ERR_UNSUPPORTED, "the next layer needs a fixed tensor scale (WQ_ACT_SCALE_STATIC): no "
                                        "output tile sees a whole row");
    if (next->cfg.rank != 0)
        return fail(WQ_ERR_UNSUPPORTED, "the next layer's low-rank branch needs its whole input row (rank must be 0)");
    if (next->device != h->device) return fail(WQ_ERR_INVALID, "handles on different devices");
    if (!x || !codes || !scales_mma || !gscale || !workspace || (next->cfg.n_outliers && !x_omega))
        return fail(WQ_ERR_INVALID, "NULL buffer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(scales_mma) |
         reinterpret_cast<uintptr_t>(x_omega)) & 15)
        return fail(WQ_ERR_INVALID, "device buffers must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(WQ_ERR_INVALID, "workspace must be 256-byte aligned");
    if (const wq_status d = check_device(h)) return d;
    const wq::ActWorkspace ws = wq::carve_workspace(workspace, M, h->cfg.K, h->r_pad, h->no_pad);
    if (workspace_bytes < ws.bytes) return fail(WQ_ERR_INVALID, "workspace too small");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    wq_status s = run_quant(h, x, M, WQ_SCALE_LAYOUT_MMA, ws.codes, ws.sf, ws.g, h->no_pad ? ws.xo : nullptr,
                            h->r_pad ? ws.u : nullptr, ws.amax, st);
    if (s != WQ_OK) return s;
    wq::ChainArgs c{};
    c.inv_s = next->d_inv_s;
    c.rotate = next->cfg.rotate | (next->cfg.rotate && next->cfg.transform_order == WQ_ORDER_ROTATE_SMOOTH ? 2 : 0);
    c.omega_blk = next->d_omega_blk;
    c.n_out = next->cfg.n_outliers;
    c.xo_ld = next->no_pad;
    c.xo = static_cast<uint16_t*>(x_omega);
    c.codes = codes;
    c.sf = scales_mma;
    c.g_out = gscale;
    c.g = next->cfg.act_gscale;
    // the output map is never used in this mode; it is keyed to the codes buffer
    return run_gemm(h, ws.codes, ws.sf, ws.g, ws.u, ws.xo, M, codes, st, &c);
}

WQ_API wq_status wq_linear_forward_quantized(wq_weights_t h, const uint8_t* codes, const uint8_t* scales_mma,
                                             const float* gscale, const void* u, const void* x_omega, int M,
                                             void* y, void* stream) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    if (M == 0) return WQ_OK;
    const bool w8 = h->cfg.mode != WQ_MODE_W4A4;
    if (!codes || (!scales_mma && !w8) || !gscale || !y) return fail(WQ_ERR_INVALID, "NULL buffer");
    if (h->cfg.rank > 0 && !u) return fail(WQ_ERR_INVALID, "u is required when rank > 0");
    if (h->cfg.n_outliers > 0 && !x_omega) return fail(WQ_ERR_INVALID, "x_omega is required when n_outliers > 0");
    if ((reinterpret_cast<uintptr_t>(codes) | reinterpret_cast<uintptr_t>(scales_mma) |
         reinterpret_cast<uintptr_t>(u) | reinterpret_cast<uintptr_t>(x_omega) | reinterpret_cast<uintptr_t>(y)) & 15)
        return fail(WQ_ERR_INVALID, "device buffers must be 16-byte aligned");
    if (const wq_status d = check_device(h)) return d;
    return run_gemm(h, codes, scales_mma, gscale, static_cast<const uint16_t*>(u),
                    static_cast<const uint16_t*>(x_omega), M, y, static_cast<cudaStream_t>(stream));
}

WQ_API wq_status wq_linear_forward_w8a8(wq_weights_t h, const void* x, int M, void* y, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (h->cfg.mode != WQ_MODE_W8A8 && h->cfg.mode != WQ_MODE_W8A8_FP8)
        return fail(WQ_ERR_INVALID, "handle was not prepared with an 8-bit weight mode");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    if (M == 0) return WQ_OK;
    if (!x || !y || !workspace) return fail(WQ_ERR_INVALID, "NULL buffer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15)
        return fail(WQ_ERR_INVALID, "x and y must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return fail(WQ_ERR_INVALID, "workspace must be 256-byte aligned");
    if (const wq_status d = check_device(h)) return d;
    if (workspace_bytes < w8_workspace_bytes(h, M)) return fail(WQ_ERR_INVALID, "workspace too small");
    uint8_t* codes = static_cast<uint8_t*>(workspace);
    float* a = reinterpret_cast<float*>(codes + align_up(w8_code_bytes(h, M), 1024));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    wq_status s = run_quant(h, x, M, WQ_SCALE_LAYOUT_ROWMAJOR, codes, nullptr, a, nullptr, nullptr, nullptr, st);
    if (s != WQ_OK) return s;
    return run_gemm(h, codes, nullptr, a, nullptr, nullptr, M, y, st);
}

WQ_API wq_status wq_quantize_activations_w8a8(wq_weights_t h, const void* x, int M, void* codes, float* scale,
                                              void* stream) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (h->cfg.mode != WQ_MODE_W8A8 && h->cfg.mode != WQ_MODE_W8A8_FP8)
        return fail(WQ_ERR_INVALID, "handle was not prepared with an 8-bit weight mode");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    if (M == 0) return WQ_OK;
    if (!x || !codes || !scale) return fail(WQ_ERR_INVALID, "NULL buffer");
    if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(codes)) & 15)
        return fail(WQ_ERR_INVALID, "device buffers must be 16-byte aligned");
    if (const wq_status d = check_device(h)) return d;
    return run_quant(h, x, M, WQ_SCALE_LAYOUT_ROWMAJOR, static_cast<uint8_t*>(codes), nullptr, scale, nullptr,
                     nullptr, nullptr, static_cast<cudaStream_t>(stream));
}

WQ_API wq_status wq_export_weights_w8a8(wq_weights_t h, int8_t* q, float* w) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (h->cfg.mode != WQ_MODE_W8A8 && h->cfg.mode != WQ_MODE_W8A8_FP8)
        return fail(WQ_ERR_INVALID, "handle was not prepared with an 8-bit weight mode");
    const int K = h->cfg.K, N = h->cfg.N;
    if (q && h->cfg.mode == WQ_MODE_W8A8_FP8) {
        WQ_CUDA(cudaMemcpy(q, h->d_codes, static_cast<size_t>(N) * K, cudaMemcpyDeviceToHost), "export");
    } else if (q) {
        std::vector<uint16_t> b(static_cast<size_t>(N) * K);
        WQ_CUDA(cudaMemcpy(b.data(), h->d_codes, b.size() * 2, cudaMemcpyDeviceToHost), "export");
        for (size_t i = 0; i < b.size(); ++i)
            q[i] = static_cast<int8_t>(__bfloat162float(__ushort_as_bfloat16(b[i])));
    }
    if (w) WQ_CUDA(cudaMemcpy(w, h->d_colscale, static_cast<size_t>(N) * 4, cudaMemcpyDeviceToHost), "export");
    return WQ_OK;
}

WQ_API wq_status wq_prepare_conv3d(const float* w, int C_in, int C_out, int kt, int kh, int kw, int pad, void* stream,
                                   wq_weights_t* out) {
    g_last_error.clear();
    if (!out) return fail(WQ_ERR_INVALID, "out is NULL");
    *out = nullptr;
    if (!w) return fail(WQ_ERR_INVALID, "w is NULL");
    if (C_in <= 0 || C_out <= 0) return fail(WQ_ERR_INVALID, "channel counts must be positive");
    if (kt <= 0 || kh <= 0 || kw <= 0 || pad < 0) return fail(WQ_ERR_INVALID, "bad kernel extent or padding");
    if (kt != 3 || kh != 3 || kw != 3 || pad != 1)
        return fail(WQ_ERR_UNSUPPORTED, "the implicit GEMM implements a 3 x 3 x 3 kernel with padding 1");
    if (C_in % 128 || C_out % 16 || 27 * C_in > 16384)
        return fail(WQ_ERR_UNSUPPORTED, "need C_in % 128 == 0, C_out % 16 == 0 and 27 C_in <= 16384");
    const int K = 27 * C_in, N = C_out;
    std::vector<float> Wm(static_cast<size_t>(K) * N);      // [K = (kd, kh, kw, c_in), N]
    for (int n = 0; n < N; ++n)
        for (int c = 0; c < C_in; ++c)
            for (int t = 0; t < 27; ++t)
                Wm[(static_cast<size_t>(t) * C_in + c) * N + n] = w[(static_cast<size_t>(n) * C_in + c) * 27 + t];
    wq_config cfg{K, N, 0, 0, 0, WQ_MODE_W4A4, WQ_ACT_SCALE_ROW, 0.0f, WQ_ORDER_SMOOTH_ROTATE, 0};
    wq_weights_t h = nullptr;
    const wq_status st = wq_prepare_weights(&cfg, Wm.data(), nullptr, nullptr, nullptr, nullptr, nullptr, stream, &h);
    if (st != WQ_OK) return st;
    h->conv_cin = C_in;
    const char* why = "";
    if (!wq::encode_tmap_2d(&h->tmBconv, CU_TENSOR_MAP_DATA_TYPE_UINT8, h->d_codes, K / 2, N, K / 2, 64, 128,
                            CU_TENSOR_MAP_SWIZZLE_64B, &why)) {
        wq_free_weights(h);
        return fail(WQ_ERR_CUDA, why);
    }
    *out = h;
    return WQ_OK;
}

WQ_API size_t wq_conv3d_workspace_bytes(wq_weights_t h, int B, int D, int H, int W) {
    if (!h || h->conv_cin == 0 || B <= 0 || D <= 0 || H <= 0 || W <= 0) return 0;
    return wq::conv_workspace_bytes(h->conv_cin, B * D * H * W, h->num_sms);
}

static wq_status conv_args(wq_weights_t h, const void* x, int B, int D, int H, int W, void* ws, size_t ws_bytes,
                           wq::ConvArgs* a) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (h->conv_cin == 0) return fail(WQ_ERR_INVALID, "handle was not prepared with wq_prepare_conv3d");
    if (!x || !ws) return fail(WQ_ERR_INVALID, "NULL buffer");
    if (B <= 0 || D <= 0 || H <= 0 || W <= 0) return fail(WQ_ERR_INVALID, "bad batch or spatial size");
    if ((D * H * W) % 8) return fail(WQ_ERR_UNSUPPORTED, "D H W must be a multiple of 8");
    if (static_cast<long long>(B) * D * H * W * h->conv_cin >= (1ll << 31))
        return fail(WQ_ERR_UNSUPPORTED, "the input must have fewer than 2^31 elements");
    const int V = B * D * H * W;
    if ((reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(ws) & 255))
        return fail(WQ_ERR_INVALID, "x must be 16-byte and the workspace 256-byte aligned");
    if (ws_bytes < wq_conv3d_workspace_bytes(h, B, D, H, W)) return fail(WQ_ERR_INVALID, "workspace too small");
    if (const wq_status d = check_device(h)) return d;
    const int C = h->conv_cin;
    uint8_t* b = static_cast<uint8_t*>(ws);
    auto al = [](size_t v) { return (v + 1023) / 1024 * 1024; };
    a->x = x; a->C = C; a->D = D; a->H = H; a->W = W; a->V = V; a->N = h->cfg.N;
    a->partial = reinterpret_cast<float*>(b);
    a->g = a->partial + 2 * h->num_sms;
    a->codes = b + al(static_cast<size_t>(2 * h->num_sms + 1) * 4);
    a->scales = a->codes + al(static_cast<size_t>(V) * C / 2);
    a->tmB = &h->tmBconv; a->sfb = h->d_sf; a->gw = h->gW; a->err = h->d_err; a->num_sms = h->num_sms;
    return WQ_OK;
}

WQ_API wq_status wq_conv3d_forward(wq_weights_t h, const void* x, int B, int D, int H, int W, void* y,
                                   void* workspace, size_t workspace_bytes, void* stream) {
    wq::ConvArgs a{};
    wq_status s = conv_args(h, x, B, D, H, W, workspace, workspace_bytes, &a);
    if (s != WQ_OK) return s;
    if (!y || (reinterpret_cast<uintptr_t>(y) & 15)) return fail(WQ_ERR_INVALID, "y must be a 16-byte aligned buffer");
    a.y = y;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = wq::launch_conv_quant(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "conv quantiser launch");
    e = wq::launch_conv_gemm(a, st);
    if (e != cudaSuccess) return cuda_fail(e, "conv GEMM launch");
    return WQ_OK;
}

WQ_API wq_status wq_quantize_conv3d_input(wq_weights_t h, const void* x, int B, int D, int H, int W, uint8_t* codes,
                                          uint8_t* scales, float* g, void* workspace, size_t workspace_bytes,
                                          void* stream) {
    wq::ConvArgs a{};
    wq_status s = conv_args(h, x, B, D, H, W, workspace, workspace_bytes, &a);
    if (s != WQ_OK) return s;
    if (!codes || !scales || !g) return fail(WQ_ERR_INVALID, "NULL output");
    if ((reinterpret_cast<uintptr_t>(codes) & 15) || (reinterpret_cast<uintptr_t>(scales) & 3))
        return fail(WQ_ERR_INVALID, "codes must be 16-byte and scales 4-byte aligned");
    a.codes = codes; a.scales = scales; a.g = g;
    const cudaError_t e = wq::launch_conv_quant(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "conv quantiser launch");
    return WQ_OK;
}

WQ_API wq_status wq_linear_forward_host(wq_weights_t h, const void* x_host, int M, void* y_host, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (M < 0) return fail(WQ_ERR_INVALID, "M < 0");
    if (M == 0) return WQ_OK;
    if (!x_host || !y_host || !workspace) return fail(WQ_ERR_INVALID, "NULL buffer");
    if (workspace_bytes < wq_host_workspace_bytes(h, M)) return fail(WQ_ERR_INVALID, "workspace too small");
    if (const wq_status d = check_device(h)) return d;
    const size_t wsb = wq_workspace_bytes(h, M);
    const int K = h->cfg.K, N = h->cfg.N;
    const size_t xb = static_cast<size_t>(M) * K * 2;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    uint8_t* dx = base + wsb;
    uint8_t* dy = base + wsb + align_up(xb, 1024);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const bool eight = h->cfg.mode == WQ_MODE_W8A8 || h->cfg.mode == WQ_MODE_W8A8_FP8;
    auto forward = [&](const void* xd, int rows, void* yd) {
        const size_t w = wq_workspace_bytes(h, rows);
        return eight ? wq_linear_forward_w8a8(h, xd, rows, yd, workspace, w, stream)
                     : wq_linear_forward(h, xd, rows, yd, workspace, w, stream);
    };
    // Row chunks of at least 2048 rows (at most 8): chunk c's upload (copy_in), forward (`stream`)
    // and download (copy_out) are ordered by events, so the copies of different chunks overlap
    // each other and the kernels, in both directions at once.  The uploads start after the work
    // queued on `stream` before this call, and `stream` resumes only after the last download.
    const int nch = std::max(1, std::min(8, M / 2048));
    if (nch == 1) {
        WQ_CUDA(cudaMemcpyAsync(dx, x_host, xb, cudaMemcpyHostToDevice, st), "x upload");
        const wq_status s = forward(dx, M, dy);
        if (s != WQ_OK) return s;
        WQ_CUDA(cudaMemcpyAsync(y_host, dy, static_cast<size_t>(M) * N * 2, cudaMemcpyDeviceToHost, st), "y download");
        return WQ_OK;
    }
    const int rows_per = static_cast<int>(align_up(static_cast<size_t>((M + nch - 1) / nch), 256));
    std::lock_guard<std::mutex> lk(h->mu_host);
    if (!h->copy_in) WQ_CUDA(cudaStreamCreateWithFlags(&h->copy_in, cudaStreamNonBlocking), "copy stream");
    if (!h->copy_out) WQ_CUDA(cudaStreamCreateWithFlags(&h->copy_out, cudaStreamNonBlocking), "copy stream");
    while (h->host_events.size() < 2u * 8u + 2u) {
        cudaEvent_t e;
        WQ_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "event");
        h->host_events.push_back(e);
    }
    cudaEvent_t* ev = h->host_events.data();            // [0] start, [1] end, [2 + 2c] in, [3 + 2c] out
    WQ_CUDA(cudaEventRecord(ev[0], st), "event");
    WQ_CUDA(cudaStreamWaitEvent(h->copy_in, ev[0], 0), "event wait");
    WQ_CUDA(cudaStreamWaitEvent(h->copy_out, ev[0], 0), "event wait");
    const uint8_t* xh = static_cast<const uint8_t*>(x_host);
    uint8_t* yh = static_cast<uint8_t*>(y_host);
    for (int c = 0, r0 = 0; r0 < M; ++c, r0 += rows_per) {
        const int rows = std::min(rows_per, M - r0);
        const size_t xo = static_cast<size_t>(r0) * K * 2, yo = static_cast<size_t>(r0) * N * 2;
        WQ_CUDA(cudaMemcpyAsync(dx + xo, xh + xo, static_cast<size_t>(rows) * K * 2, cudaMemcpyHostToDevice, h->copy_in),
                "x upload");
        WQ_CUDA(cudaEventRecord(ev[2 + 2 * c], h->copy_in), "event");
        WQ_CUDA(cudaStreamWaitEvent(st, ev[2 + 2 * c], 0), "event wait");
        const wq_status s = forward(dx + xo, rows, dy + yo);
        if (s != WQ_OK) return s;
        WQ_CUDA(cudaEventRecord(ev[3 + 2 * c], st), "event");
        WQ_CUDA(cudaStreamWaitEvent(h->copy_out, ev[3 + 2 * c], 0), "event wait");
        WQ_CUDA(cudaMemcpyAsync(yh + yo, dy + yo, static_cast<size_t>(rows) * N * 2, cudaMemcpyDeviceToHost, h->copy_out),
                "y download");
    }
    WQ_CUDA(cudaEventRecord(ev[1], h->copy_out), "event");
    WQ_CUDA(cudaStreamWaitEvent(st, ev[1], 0), "event wait");
    return WQ_OK;
}

WQ_API wq_status wq_export_weights(wq_weights_t h, uint8_t* codes, uint8_t* scales, float* gW, uint16_t* P,
                                   uint16_t* Q, uint16_t* W_omega) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (h->cfg.mode != WQ_MODE_W4A4 && h->cfg.mode != WQ_MODE_W4A8)
        return fail(WQ_ERR_INVALID, "W8A8 handle: use wq_export_weights_w8a8");
    const int K = h->cfg.K, N = h->cfg.N, r = h->cfg.rank, no = h->cfg.n_outliers;
    const int rp = h->r_pad, nop = h->no_pad;
    if (codes) WQ_CUDA(cudaMemcpy(codes, h->d_codes, static_cast<size_t>(N) * K / 2, cudaMemcpyDeviceToHost), "export");
    if (scales) {
        const size_t n_pad = align_up(static_cast<size_t>(N), wq::kBlockM);
        std::vector<uint8_t> sf(n_pad / wq::kBlockM * (K / 64) * wq::kSfAtom);
        WQ_CUDA(cudaMemcpy(sf.data(), h->d_sf, sf.size(), cudaMemcpyDeviceToHost), "export");
        for (int n = 0; n < N; ++n)
            for (int b = 0; b < K / 16; ++b)
                scales[static_cast<size_t>(n) * (K / 16) + b] =
                    sf[((static_cast<size_t>(n) / 128) * (K / 64) + b / 4) * wq::kSfAtom + (n % 32) * 16 +
                       ((n % 128) / 32) * 4 + (b % 4)];
    }
    if (gW) *gW = h->gW;
    if (P && r) {
        std::vector<uint16_t> pp(static_cast<size_t>(K) * rp);
        WQ_CUDA(cudaMemcpy(pp.data(), h->d_P, pp.size() * 2, cudaMemcpyDeviceToHost), "export");
        for (int k = 0; k < K; ++k)
            for (int j = 0; j < r; ++j) P[static_cast<size_t>(k) * r + j] = pp[static_cast<size_t>(k) * rp + j];
    }
    if (Q && r) {
        std::vector<uint16_t> qt(static_cast<size_t>(N) * rp);
        WQ_CUDA(cudaMemcpy(qt.data(), h->d_Qt, qt.size() * 2, cudaMemcpyDeviceToHost), "export");
        for (int n = 0; n < N; ++n)
            for (int j = 0; j < r; ++j) Q[static_cast<size_t>(j) * N + n] = qt[static_cast<size_t>(n) * rp + j];
    }
    if (W_omega && no) {
        std::vector<uint16_t> wt(static_cast<size_t>(N) * nop);
        WQ_CUDA(cudaMemcpy(wt.data(), h->d_WOt, wt.size() * 2, cudaMemcpyDeviceToHost), "export");
        for (int n = 0; n < N; ++n)
            for (int j = 0; j < no; ++j) W_omega[static_cast<size_t>(j) * N + n] = wt[static_cast<size_t>(n) * nop + j];
    }
    return WQ_OK;
}

WQ_API wq_status wq_check_device_error(wq_weights_t h, void* stream) {
    if (!h) return fail(WQ_ERR_INVALID, "NULL handle");
    if (const wq_status d = check_device(h)) return d;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    WQ_CUDA(cudaStreamSynchronize(st), "stream synchronise");
    int v = 0;
    WQ_CUDA(cudaMemcpy(&v, h->d_err, sizeof(int), cudaMemcpyDeviceToHost), "error flag read");
    if (v != 0) {
        WQ_CUDA(cudaMemset(h->d_err, 0, sizeof(int)), "error flag clear");
        return fail(WQ_ERR_TIMEOUT, "kernel barrier wait timed out (site " + std::to_string(v) + ")");
    }
    return WQ_OK;
}

WQ_API void wq_free_weights(wq_weights_t h) {
    if (!h) return;
    cudaDeviceSynchronize();
    free_device(h);
    delete h;
}

}  // extern "C"
