// Host side of the tcgen05 prefill GEMM: tile geometry, tensor maps and
// dispatch.  bf16 activations run the hi/lo kernel (gemm_hl.cuh: the weight
// as an exact-enough sum of two bf16 values, one accumulator); f16
// activations run the block-scaled kernel (gemm_bs.cuh: exact (q - zp) and
// one TMEM partial per quantisation block), whose f32 rescale has no range
// limit where an f16 weight would.  MNB_TC_KERNEL=bs forces the latter.
#include <cstdio>
#include <cstdlib>
#include <cstring>

#include "gemm_bs.cuh"
#include "gemm_hl.cuh"

namespace mnb {
cudaError_t launch_gemm_tc_b2(const MatmulParams& p, const gbs::Geom& geo, const gbs::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_tc_b4(const MatmulParams& p, const gbs::Geom& geo, const gbs::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_tc_b8(const MatmulParams& p, const gbs::Geom& geo, const gbs::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_a8_b2(const MatmulParams& p, const ghl::Geom& geo, const ghl::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_a8_b4(const MatmulParams& p, const ghl::Geom& geo, const ghl::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_a8_b8(const MatmulParams& p, const ghl::Geom& geo, const ghl::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_hl_b2(const MatmulParams& p, const ghl::Geom& geo, const ghl::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_hl_b4(const MatmulParams& p, const ghl::Geom& geo, const ghl::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_hl_b8(const MatmulParams& p, const ghl::Geom& geo, const ghl::Maps& m, cudaStream_t s);

namespace {
using gbs::Geom;
using gbs::Maps;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return (EncodeTiledFn) nullptr;
        }
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

// Tokens per tile BT in {32, 64, 128} (at most max_bt): fewest waves of
// (128-row x BT) tiles over the SMs, then the least padded work; MNB_TC_BT
// forces one.
Geom make_geom(const MatmulParams& p, int max_bt = 128) {
    Geom g{};
    const Layout& L = p.L;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    const int64_t nt = (L.N + gbs::kRows - 1) / gbs::kRows;
    const char* env = std::getenv("MNB_TC_BT");
    const int forced = env ? std::atoi(env) : 0;
    double best = 1e30;
    for (int bt = 32; bt <= max_bt; bt *= 2) {
        if (forced && bt != forced) continue;
        const int64_t mt = (p.M + bt - 1) / bt;
        const int64_t waves = (nt * mt + sms - 1) / sms;
        // per-SM cost of a wave ~ BT token columns plus a fixed per-tile cost
        // (pipeline fill, epilogue) worth about 32 columns
        const double cost = (double)waves * (bt + 32) + 1e-3 * (double)(mt * bt - p.M);
        if (cost < best) {
            best = cost;
            g.BT = bt;
        }
    }
    if (g.BT == 0) g.BT = max_bt;
    g.n_tiles = (int)nt;
    g.m_tiles = (int)((p.M + g.BT - 1) / g.BT);
    g.k_stages = (int)((L.Kpad + gbs::kBK - 1) / gbs::kBK);
    g.x_stage = (size_t)g.BT * gbs::kBK * 2;
    g.wp_stage = (size_t)(gbs::kRows / 16) * (gbs::kBK / L.KT) * kTileBytes;
    const size_t fixed = 1024 + gbs::kBarBytes;
    const size_t limit = device_info().smem_optin ? device_info().smem_optin : 232448;
    g.R = gbs::kMaxR;
    while (g.R > 2 && fixed + g.R * (g.x_stage + g.wp_stage) > limit) --g.R;
    g.NP = (512 - g.R * gbs::kACols) / g.BT;
    if (g.NP > gbs::kMaxNP) g.NP = gbs::kMaxNP;
    g.a_col0 = g.NP * g.BT;
    g.tmem_cols = 32;
    while (g.tmem_cols < g.a_col0 + g.R * gbs::kACols) g.tmem_cols <<= 1;
    g.total_bytes = fixed + g.R * (g.x_stage + g.wp_stage);
    return g;
}

// Tensor maps of the block-scaled kernel: X [M][xk] (bf16 / f16, row stride
// xk * 2 bytes), 64-deep x BT-token boxes, 128-byte swizzle, zero fill past M
// and xk; the packed codes, each 512-byte tile loaded as [chunk t][row group
// g][16 B] (dims: 8 x u16, g (stride 64 B), t (stride 16 B), k tile, row tile).
cudaError_t make_bs_maps(const MatmulParams& p, const Geom& geo, EncodeTiledFn enc, const void* x, int64_t xk,
                         int x_dtype, Maps* m) {
    std::memset(m, 0, sizeof(*m));
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {(cuuint64_t)xk, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)xk * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)geo.BT};
    const CUtensorMapDataType dt =
        x_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(&m->x, dt, 2, const_cast<void*>(x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    const cuuint64_t tdims[5] = {8, 8, 4, (cuuint64_t)p.L.KTILES, (cuuint64_t)p.L.NT};
    const cuuint64_t tstrides[4] = {64, 16, (cuuint64_t)kTileBytes, (cuuint64_t)p.L.KTILES * kTileBytes};
    const cuuint32_t tbox[5] = {8, 8, 4, (cuuint32_t)(gbs::kBK / p.L.KT), (cuuint32_t)(gbs::kRows / 16)};
    const cuuint32_t testr[5] = {1, 1, 1, 1, 1};
    r = enc(&m->w, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<uint8_t*>(p.packed), tdims, tstrides, tbox, testr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (std::getenv("MNB_LOG")) std::fprintf(stderr, "[mnb] 5-D code map rejected (%d)\n", (int)r);
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

bool use_hl(const MatmulParams& p) {
    const char* k = std::getenv("MNB_TC_KERNEL");
    if (k && std::strcmp(k, "bs") == 0) return false;
    return p.act_dtype == kBF16;
}

// hi/lo kernel: 128 W rows x 256 tokens per tile; the two CTAs of a cluster
// split K when one tile per CTA would leave more than half the SMs idle.
// tf32: the accuracy level 4 variant (f32 X stages of 64 KB, a ring of three).
ghl::Geom make_geom_hl(const MatmulParams& p, bool tf32 = false) {
    ghl::Geom g{};
    const Layout& L = p.L;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    g.n_tiles = (int)((L.N + ghl::kRows - 1) / ghl::kRows);
    g.m_tiles = (int)((p.M + ghl::kBT - 1) / ghl::kBT);
    g.k_stages = (int)((L.Kpad + ghl::kBK - 1) / ghl::kBK);
    const int64_t tiles = (int64_t)g.n_tiles * g.m_tiles;
    g.splitk = (2 * tiles <= sms && g.k_stages >= 2) ? 2 : 1;
    const char* env = std::getenv("MNB_TC_SPLITK");
    if (env && (env[0] == '1' || env[0] == '2')) g.splitk = (env[0] == '2' && g.k_stages >= 2) ? 2 : 1;
    const int tiles_per_stage = L.KT >= ghl::kBK ? 1 : (int)(ghl::kBK / L.KT);
    g.wp_stage = (size_t)(ghl::kRows / 16) * tiles_per_stage * kTileBytes;
    const int R = tf32 ? 3 : ghl::kR;
    const size_t xst = tf32 ? 2 * (size_t)ghl::kXStage : (size_t)ghl::kXStage;
    g.total_bytes = 1024 + R * (xst + g.wp_stage) + ghl::hl_bar_bytes(R);
    return g;
}

// The packed codes of the hi/lo and tf32 kernels: each 512-byte tile as [chunk
// t][row group g][16 B], one stage's tiles of 128 rows per box.
CUresult hl_wmap(const MatmulParams& p, EncodeTiledFn enc, CUtensorMap* w) {
    const cuuint64_t tdims[5] = {8, 8, 4, (cuuint64_t)p.L.KTILES, (cuuint64_t)p.L.NT};
    const cuuint64_t tstrides[4] = {64, 16, (cuuint64_t)kTileBytes, (cuuint64_t)p.L.KTILES * kTileBytes};
    const cuuint32_t tbox[5] = {8, 8, 4, (cuuint32_t)(p.L.KT >= ghl::kBK ? 1 : ghl::kBK / p.L.KT),
                                (cuuint32_t)(ghl::kRows / 16)};
    const cuuint32_t testr[5] = {1, 1, 1, 1, 1};
    return enc(w, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<uint8_t*>(p.packed), tdims, tstrides, tbox, testr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

// Y for the TMA store of the hi/lo and tf32 kernels: [M][N] of out_dtype, boxes of
// 128 bytes of rows x the CTA's tokens (256, or 128 with a K split).  False
// (element stores instead) when Y's base or row stride is not 16-byte aligned.
bool hl_ymap(const MatmulParams& p, const ghl::Geom& geo, EncodeTiledFn enc, CUtensorMap* y) {
    const int es = p.out_dtype == kF32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(p.y) & 15) != 0 || (p.L.N * es) % 16 != 0) return false;
    const CUtensorMapDataType dt = p.out_dtype == kF32   ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : p.out_dtype == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const cuuint64_t dims[2] = {(cuuint64_t)p.L.N, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.L.N * es};
    const cuuint32_t box[2] = {(cuuint32_t)(128 / es), (cuuint32_t)(geo.splitk == 2 ? ghl::kBT / 2 : ghl::kBT)};
    const cuuint32_t estr[2] = {1, 1};
    return enc(y, dt, 2, p.y, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_hl(const MatmulParams& p, EncodeTiledFn enc, cudaStream_t s) {
    ghl::Geom geo = make_geom_hl(p);
    ghl::Maps m;
    std::memset(&m, 0, sizeof(m));
    geo.ystore = hl_ymap(p, geo, enc, &m.y) ? 1 : 0;
    geo.pdl = (p.flags & kFlagPDL) ? 1 : 0;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {(cuuint64_t)p.L.K, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.L.K * 2};
    const cuuint32_t box[2] = {ghl::kBK, ghl::kBT};
    CUresult r = enc(&m.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.x), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (hl_wmap(p, enc, &m.w) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    switch (p.L.bits) {
        case 2: return launch_gemm_hl_b2(p, geo, m, s);
        case 4: return launch_gemm_hl_b4(p, geo, m, s);
        case 8: return launch_gemm_hl_b8(p, geo, m, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool gemm_tc_supported(const MatmulParams& p) {
    if (p.g_idx != nullptr || p.M < 1) return false;
    if (p.act_dtype != kBF16 && p.act_dtype != kF16) return false;
    const DeviceInfo& di = device_info();
    if (di.major != 10) return false;                   // tcgen05 needs the sm_100 family
    if ((p.L.K * 2) % 16 != 0) return false;            // TMA row stride of X
    if ((reinterpret_cast<uintptr_t>(p.x) & 15) != 0) return false;
    if (p.L.K > (int64_t)1 << 31 || p.M > (int64_t)1 << 31) return false;
    if (!encode_fn()) return false;
    if (use_hl(p)) {
        const ghl::Geom h = make_geom_hl(p);
        return h.total_bytes <= di.smem_optin && (int64_t)h.n_tiles * h.m_tiles * h.splitk < (int64_t)1 << 31;
    }
    const Geom g = make_geom(p);
    return g.NP >= 2 && g.total_bytes <= di.smem_optin && (int64_t)g.n_tiles * g.m_tiles < (int64_t)1 << 31;
}

cudaError_t launch_gemm_tc(const MatmulParams& p, cudaStream_t s) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    if (use_hl(p)) return launch_hl(p, enc, s);
    const Geom geo = make_geom(p);
    Maps m;
    const cudaError_t me = make_bs_maps(p, geo, enc, p.x, p.L.K, p.act_dtype, &m);
    if (me != cudaSuccess) return me;
    switch (p.L.bits) {
        case 2: return launch_gemm_tc_b2(p, geo, m, s);
        case 4: return launch_gemm_tc_b4(p, geo, m, s);
        case 8: return launch_gemm_tc_b8(p, geo, m, s);
        default: return cudaErrorInvalidValue;
    }
}

bool gemm_a8_supported(const MatmulParams& p) {
    if (p.g_idx != nullptr || p.M < 1 || p.M > (int64_t)1 << 31 || p.L.Kpad > (int64_t)1 << 31) return false;
    const DeviceInfo& di = device_info();
    if (di.major != 10 || !encode_fn()) return false;
    const ghl::Geom g = make_geom_hl(p, true);
    return g.total_bytes <= di.smem_optin && (int64_t)g.n_tiles * g.m_tiles < (int64_t)1 << 31;
}

// Accuracy level 4 prefill: quantise X per block and write code * s_a as
// tf32 into the workspace, then the tf32 variant of the hi/lo kernel.
cudaError_t launch_gemm_a8(const MatmulParams& p, cudaStream_t s) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    float* xq = static_cast<float*>(p.workspace);
    cudaError_t e = launch_quant_act_tf32(p.x, p.act_dtype, xq, p.M, p.L, (p.flags & kFlagPDL) != 0, s);
    if (e != cudaSuccess) return e;
    MatmulParams q = p;
    q.x = xq;
    q.act_dtype = kF32;
    ghl::Geom geo = make_geom_hl(q, true);
    ghl::Maps m;
    std::memset(&m, 0, sizeof(m));
    geo.ystore = hl_ymap(q, geo, enc, &m.y) ? 1 : 0;
    geo.pdl = (p.flags & kFlagPDL) ? 1 : 0;
    const cuuint32_t estr[2] = {1, 1};
    const cuuint64_t dims[2] = {(cuuint64_t)p.L.Kpad, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.L.Kpad * 4};
    const cuuint32_t box[2] = {32, ghl::kBT};  // 128 bytes of depth x 256 tokens
    CUresult r = enc(&m.x, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, xq, dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS || hl_wmap(q, enc, &m.w) != CUDA_SUCCESS) return cudaErrorInvalidValue;
    switch (p.L.bits) {
        case 2: return launch_gemm_a8_b2(q, geo, m, s);
        case 4: return launch_gemm_a8_b4(q, geo, m, s);
        case 8: return launch_gemm_a8_b8(q, geo, m, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mnb
