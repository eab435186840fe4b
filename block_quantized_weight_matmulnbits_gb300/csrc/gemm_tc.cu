// Host side of the tcgen05 prefill GEMM (kernel in gemm_tc.cuh): tile
// geometry, tensor maps and dispatch to the per-code-width instantiations.
#include "gemm_ta.cuh"

namespace mnb {
cudaError_t launch_gemm_tc_b2(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_tc_b4(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_tc_b8(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_ta_b2(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_ta_b4(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s);
cudaError_t launch_gemm_ta_b8(const MatmulParams& p, const gtc::TcGeom& geo, const gtc::Maps& m, cudaStream_t s);

namespace {
using gtc::TcGeom;
using gtc::Maps;
using gtc::kBM;
using gtc::kMaxR;


typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPoint("cuTensorMapEncodeTiled", &ptr, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiledFn) nullptr;
        return reinterpret_cast<EncodeTiledFn>(ptr);
    }();
    return fn;
}

TcGeom make_geom(const MatmulParams& p) {
    TcGeom g{};
    const Layout& L = p.L;
    g.BK = L.bits == 2 ? 128 : 64;
    const int tiles = (int)(g.BK / L.KT);  // packed tiles per 16-row tile per stage: 4-bit 1, 8-bit 2, 2-bit 1
    g.m_tiles = (int)((p.M + kBM - 1) / kBM);
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    // BN (multiple of 16, <= 256): fewest waves, then least padded work
    const char* env = std::getenv("MNB_TC_BN");
    const int forced = env ? std::atoi(env) : 0;
    double best = 1e30;
    g.nbs = L.bs >= g.BK ? 1 : (int)(g.BK / L.bs);
    const int max_bn = 256 / g.nbs < 256 ? 256 / g.nbs : 256;  // entries per stage <= 256
    for (int bn = 16; bn <= max_bn; bn += 16) {
        if (forced && bn != forced) continue;
        const int64_t nt = (L.N + bn - 1) / bn;
        const int64_t ntiles = nt * g.m_tiles;
        const int64_t waves = (ntiles + sms - 1) / sms;
        // per-SM work of a wave ~ BN columns plus a fixed per-tile cost (pipeline fill,
        // epilogue, the X stream) worth about 32 columns
        const double cost = (double)waves * (bn + 32) + 1e-3 * (double)(nt * bn - L.N);
        if (cost < best) {
            best = cost;
            g.BN = bn;
        }
    }
    if (g.BN == 0) g.BN = max_bn;
    g.n_tiles = (int)((L.N + g.BN - 1) / g.BN);
    g.tmem_cols = 32;
    while (g.tmem_cols < g.BN) g.tmem_cols <<= 1;
    g.k_stages = (int)((L.KTILES * L.KT + g.BK - 1) / g.BK);
    g.units = (g.BN / 16) * tiles;
    g.x_stage = (size_t)kBM * g.BK * 2;
    g.wd_stage = (size_t)g.BN * g.BK * 2;
    g.wp_stage = (size_t)(g.BN / 16) * tiles * kTileBytes;
    g.ent_stage = round16((size_t)g.BN * g.nbs * 4);
    // raw scales by TMA: rows of scales / zero points must be 16-byte strided and aligned
    const int sbytes = p.scale_dtype == kF32 ? 4 : 2;
    g.sb = 16 / sbytes;
    if (g.sb < 128 / L.bits) g.sb = 128 / L.bits;  // zero-point box at least 16 bytes
    if (g.sb < g.nbs) g.sb = g.nbs;
    // a raw buffer spans at least kMaxR stages, so a warp never skips one
    while ((int64_t)g.sb * L.bs < (int64_t)kMaxR * g.BK) g.sb <<= 1;
    g.sb_stages = (int)((int64_t)g.sb * L.bs / g.BK);
    g.scale_tma = ((L.KB * sbytes) % 16 == 0) && ((reinterpret_cast<uintptr_t>(p.scales) & 15) == 0) &&
                  (p.zp == nullptr || ((L.zp_row % 16 == 0) && ((reinterpret_cast<uintptr_t>(p.zp) & 15) == 0)));
    // boxes no wider than the tensors they read
    if (g.sb > L.KB || (p.zp != nullptr && (int64_t)g.sb * L.bits / 8 > L.zp_row)) g.scale_tma = 0;
    if (std::getenv("MNB_TC_NO_SCALE_TMA")) g.scale_tma = 0;
    g.sraw_bytes = g.scale_tma ? round16((size_t)g.BN * g.sb * sbytes) : 0;
    g.zraw_bytes = (g.scale_tma && p.zp) ? round16((size_t)g.BN * g.sb * L.bits / 8) : 0;
    if (g.scale_tma) g.ent_stage = 0;  // constants come straight from the raw buffers
    const size_t fixed = 1024 + 2 * (g.sraw_bytes + g.zraw_bytes) + (4 * kMaxR + 3) * 8 + 16;
    const size_t per_stage = g.x_stage + g.wd_stage + g.wp_stage + g.ent_stage;
    const size_t limit = device_info().smem_optin ? device_info().smem_optin : 232448;
    g.R = kMaxR;
    const char* renv = std::getenv("MNB_TC_STAGES");
    if (renv && std::atoi(renv) >= 2 && std::atoi(renv) <= kMaxR) g.R = std::atoi(renv);
    while (g.R > 2 && fixed + g.R * per_stage > limit) --g.R;
    g.total_bytes = fixed + g.R * per_stage;
    return g;
}

// Geometry of the W-in-TMEM kernel (gemm_ta.cuh): 128 W rows x BT tokens per
// tile; needs the TMA raw-scale path, a ring of at least 5 stages (the
// dequantising warps take every 4th stage) and the A ring in tensor memory.
// Returns false when the shape is not for it.
bool make_geom_ta(const MatmulParams& p, TcGeom* out) {
    const char* env = std::getenv("MNB_TC_TA");
    if (env && env[0] == '0') return false;
    const Layout& L = p.L;
    TcGeom g = make_geom(p);
    if (!g.scale_tma) return false;
    g.ta = 1;
    // 128-deep stages; the raw-scale buffer must still span >= kMaxR stages
    g.BK = 128;
    g.k_stages = (int)((L.KTILES * L.KT + g.BK - 1) / g.BK);
    while ((int64_t)g.sb * L.bs < (int64_t)kMaxR * g.BK) g.sb <<= 1;
    g.sb_stages = (int)((int64_t)g.sb * L.bs / g.BK);
    if (g.sb > L.KB || (p.zp != nullptr && (int64_t)g.sb * L.bits / 8 > L.zp_row)) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    const int64_t nt = (L.N + gtc::kTaRows - 1) / gtc::kTaRows;
    double best = 1e30;
    int bt_best = 0;
    for (int bt = 16; bt <= 256; bt += 16) {
        const int64_t mt = (p.M + bt - 1) / bt;
        const int64_t waves = (nt * mt + sms - 1) / sms;
        const double cost = (double)waves * (bt + 32) + 1e-3 * (double)(mt * bt - p.M);
        if (cost < best) {
            best = cost;
            bt_best = bt;
        }
    }
    g.BN = bt_best;  // tokens per tile
    g.n_tiles = (int)nt;
    g.m_tiles = (int)((p.M + g.BN - 1) / g.BN);
    const int tiles = (int)(g.BK / L.KT);
    const int a_cols = (g.BK / 16) * 8;
    g.a_col0 = (g.BN + 31) & ~31;
    g.x_stage = (size_t)g.BN * g.BK * 2;
    g.wp_stage = (size_t)(gtc::kTaRows / 16) * tiles * kTileBytes;
    g.wd_stage = 0;
    g.ent_stage = 0;
    const int sbytes = p.scale_dtype == kF32 ? 4 : 2;
    g.sraw_bytes = round16((size_t)gtc::kTaRows * g.sb * sbytes);
    g.zraw_bytes = p.zp ? round16((size_t)gtc::kTaRows * g.sb * L.bits / 8) : 0;
    const size_t fixed = 1024 + 2 * (g.sraw_bytes + g.zraw_bytes) + (4 * kMaxR + 3) * 8 + 16;
    const size_t per_stage = g.x_stage + g.wp_stage;
    const size_t limit = device_info().smem_optin ? device_info().smem_optin : 232448;
    g.R = kMaxR;
    while (g.R > 2 && (fixed + g.R * per_stage > limit || g.a_col0 + g.R * a_cols > 512)) --g.R;
    if (g.R < 2 || g.sb_stages < g.R) return false;
    g.tmem_cols = 32;
    while (g.tmem_cols < g.a_col0 + g.R * a_cols) g.tmem_cols <<= 1;
    g.total_bytes = fixed + g.R * per_stage;
    *out = g;
    return true;
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
    const TcGeom g = make_geom(p);
    return g.total_bytes <= di.smem_optin && (int64_t)g.n_tiles * g.m_tiles < (int64_t)1 << 31;
}

cudaError_t launch_gemm_tc(const MatmulParams& p, cudaStream_t s) {
    TcGeom geo;
    if (!make_geom_ta(p, &geo)) geo = make_geom(p);
    const int rows = geo.ta ? gtc::kTaRows : geo.BN;  // W rows per tile
    EncodeTiledFn enc = encode_fn();
    if (!enc) return cudaErrorNotSupported;
    Maps m;
    std::memset(&m, 0, sizeof(m));
    const cuuint32_t estr[3] = {1, 1, 1};
    // X: [M][K] bf16/f16, 128-row x 64-deep boxes, 128-byte swizzle, zero fill past M and K
    const cuuint64_t dims[2] = {(cuuint64_t)p.L.K, (cuuint64_t)p.M};
    const cuuint64_t strides[1] = {(cuuint64_t)p.L.K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)(geo.ta ? geo.BN : kBM)};
    const CUtensorMapDataType dt =
        p.act_dtype == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    CUresult r = enc(&m.x, dt, 2, const_cast<void*>(p.x), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    // Packed codes as a 3-D tensor of 16-bit elements: [row tile][k tile][256 x u16].
    const cuuint64_t wdims[3] = {256, (cuuint64_t)p.L.KTILES, (cuuint64_t)p.L.NT};
    const cuuint64_t wstrides[2] = {(cuuint64_t)kTileBytes, (cuuint64_t)p.L.KTILES * kTileBytes};
    const cuuint32_t wbox[3] = {256, (cuuint32_t)(geo.BK / p.L.KT), (cuuint32_t)(rows / 16)};
    r = enc(&m.w, CU_TENSOR_MAP_DATA_TYPE_UINT16, 3, const_cast<uint8_t*>(p.packed), wdims, wstrides, wbox, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
    if (geo.ta) {
        // the W-in-TMEM kernel reads codes row by row: load each 512-byte tile as
        // [t][g][16 B] (dims: 8 x u16, g (stride 64), t (stride 16), k tile, row tile)
        const cuuint64_t tdims[5] = {8, 8, 4, (cuuint64_t)p.L.KTILES, (cuuint64_t)p.L.NT};
        const cuuint64_t tstrides[4] = {64, 16, (cuuint64_t)kTileBytes, (cuuint64_t)p.L.KTILES * kTileBytes};
        const cuuint32_t tbox[5] = {8, 8, 4, (cuuint32_t)(geo.BK / p.L.KT), (cuuint32_t)(rows / 16)};
        const cuuint32_t testr[5] = {1, 1, 1, 1, 1};
        r = enc(&m.w, CU_TENSOR_MAP_DATA_TYPE_UINT16, 5, const_cast<uint8_t*>(p.packed), tdims, tstrides, tbox, testr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) {
            if (std::getenv("MNB_LOG")) std::fprintf(stderr, "[mnb] 5-D code map rejected (%d)\n", (int)r);
            return cudaErrorInvalidValue;
        }
    }
    if (geo.scale_tma) {
        // scales [N][KB] and zero points [N][zp_row] in the ORT layout, SB blocks x BN rows per box
        const int sbytes = p.scale_dtype == kF32 ? 4 : 2;
        const CUtensorMapDataType sdt = p.scale_dtype == kF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                        : p.scale_dtype == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                                : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        const cuuint64_t sdims[2] = {(cuuint64_t)p.L.KB, (cuuint64_t)p.L.N};
        const cuuint64_t sstr[1] = {(cuuint64_t)p.L.KB * sbytes};
        const cuuint32_t sbox[2] = {(cuuint32_t)geo.sb, (cuuint32_t)rows};
        r = enc(&m.s, sdt, 2, const_cast<void*>(p.scales), sdims, sstr, sbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        if (p.zp) {
            const cuuint64_t zdims[2] = {(cuuint64_t)p.L.zp_row, (cuuint64_t)p.L.N};
            const cuuint64_t zstr[1] = {(cuuint64_t)p.L.zp_row};
            const cuuint32_t zbox[2] = {(cuuint32_t)(geo.sb * p.L.bits / 8), (cuuint32_t)rows};
            r = enc(&m.z, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(p.zp), zdims, zstr, zbox, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
            if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
        }
    }
    if (geo.ta) {
        switch (p.L.bits) {
            case 2: return launch_gemm_ta_b2(p, geo, m, s);
            case 4: return launch_gemm_ta_b4(p, geo, m, s);
            case 8: return launch_gemm_ta_b8(p, geo, m, s);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (p.L.bits) {
        case 2: return launch_gemm_tc_b2(p, geo, m, s);
        case 4: return launch_gemm_tc_b4(p, geo, m, s);
        case 8: return launch_gemm_tc_b8(p, geo, m, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mnb
