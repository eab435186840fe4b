// Host side of the small-batch tensor-core GEMV: five schedules of the same
// arithmetic.  gemv_ks.cuh (the default where it applies: M <= 8, K a
// multiple of the K-chunk): one 16-warp CTA per SM,
// (row tile, K-chunk) items streamed through registers.  gemv_mma.cuh (every
// other shape): one CTA per row tile.  gemv_xr.cuh: one 16-warp CTA per SM,
// X in registers, per-warp bulk-copy rings.  gemv_pers.cuh: a persistent cp.async ring.  gemv_stream.cuh:
// persistent with register prefetch.  MNB_GEMV_SCHED=xr|tile|pers|stream
// forces one (MNB_GEMV_PERS=0/1 still selects between tile and pers).
#include <cstdlib>
#include <cstring>

#include "gemv_pers.cuh"
#include "gemv_stream.cuh"
#include "gemv_ks.cuh"
#include "gemv_xr.cuh"

namespace mnb {

cudaError_t launch_gemv_mma_b2(const MatmulParams& p, const gmma::Geom& geo, cudaStream_t s);
cudaError_t launch_gemv_mma_b4(const MatmulParams& p, const gmma::Geom& geo, cudaStream_t s);
cudaError_t launch_gemv_mma_b8(const MatmulParams& p, const gmma::Geom& geo, cudaStream_t s);
cudaError_t launch_gemv_pers_b2(const MatmulParams& p, const gpers::PGeom& geo, int grid, cudaStream_t s);
cudaError_t launch_gemv_pers_b4(const MatmulParams& p, const gpers::PGeom& geo, int grid, cudaStream_t s);
cudaError_t launch_gemv_pers_b8(const MatmulParams& p, const gpers::PGeom& geo, int grid, cudaStream_t s);
cudaError_t launch_gemv_stream_b2(const MatmulParams& p, const gstr::SGeom& geo, cudaStream_t s);
cudaError_t launch_gemv_stream_b4(const MatmulParams& p, const gstr::SGeom& geo, cudaStream_t s);
cudaError_t launch_gemv_stream_b8(const MatmulParams& p, const gstr::SGeom& geo, cudaStream_t s);
cudaError_t launch_gemv_ks_b2(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s,
                             const gks::MoeKs* moe = nullptr, bool a8 = false);
cudaError_t launch_gemv_ks_b4(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s,
                             const gks::MoeKs* moe = nullptr, bool a8 = false);
cudaError_t launch_gemv_ks_b8(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s,
                             const gks::MoeKs* moe = nullptr, bool a8 = false);
cudaError_t launch_gemv_xr_b2(const MatmulParams& p, const gxr::XGeom& geo, cudaStream_t s);
cudaError_t launch_gemv_xr_b4(const MatmulParams& p, const gxr::XGeom& geo, cudaStream_t s);
cudaError_t launch_gemv_xr_b8(const MatmulParams& p, const gxr::XGeom& geo, cudaStream_t s);

static const char* sched_env() {
    const char* v = std::getenv("MNB_GEMV_SCHED");
    return (v && *v) ? v : nullptr;
}

// The k-chunk schedule: the default unless another one is forced.
static bool ks_geom(const MatmulParams& p, gks::KGeom* out) {
    if ((reinterpret_cast<uintptr_t>(p.scales) & 15) != 0) return false;
    if (p.zp && (reinterpret_cast<uintptr_t>(p.zp) & 15) != 0) return false;
    if ((reinterpret_cast<uintptr_t>(p.x) & 3) != 0) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    return gks::make_kgeom(p.L, p.M, sms, device_info().smem_optin, p.scale_dtype == kF32 ? 4 : 2, out);
}

static bool ks_ok(const MatmulParams& p, gks::KGeom* out) {
    const char* sc = sched_env();
    if (sc && std::strcmp(sc, "ks") != 0) return false;
    if (!sc && std::getenv("MNB_GEMV_PERS")) return false;
    return ks_geom(p, out);
}

bool gemv_ks_kperm_supported(const MatmulParams& p) {
    if (p.M < 1 || p.M > 8 || p.g_idx != nullptr) return false;
    if (p.act_dtype != kBF16 && p.act_dtype != kF16) return false;
    if ((reinterpret_cast<uintptr_t>(p.x) & 15) != 0) return false;  // X copied 16 bytes at a time
    gks::KGeom kg;
    if (!ks_geom(p, &kg)) return false;
    return kg.x_bytes + kg.red_bytes + gks::kperm_x_bytes(p.L, p.M) <= device_info().smem_optin;
}

cudaError_t launch_gemv_ks_kperm(const MatmulParams& p, cudaStream_t s) {
    gks::KGeom kg;
    if (!gemv_ks_kperm_supported(p) || !ks_geom(p, &kg)) return cudaErrorNotSupported;
    switch (p.L.bits) {
        case 2: return launch_gemv_ks_b2(p, kg, s);
        case 4: return launch_gemv_ks_b4(p, kg, s);
        case 8: return launch_gemv_ks_b8(p, kg, s);
        default: return cudaErrorInvalidValue;
    }
}

// The register-X schedule (opt-in with MNB_GEMV_SCHED=xr; measured slower
// than the per-tile grid on GB300: 27.5 vs 10.5 us on the int4 4096 x 11008
// decode).
static bool xr_ok(const MatmulParams& p, gxr::XGeom* out) {
    const char* sc = sched_env();
    if (!sc || std::strcmp(sc, "xr") != 0) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    const int sbytes = p.scale_dtype == kF32 ? 4 : 2;
    const bool aligned = (reinterpret_cast<uintptr_t>(p.scales) & 15) == 0 &&
                         (p.zp == nullptr || (reinterpret_cast<uintptr_t>(p.zp) & 15) == 0);
    return gxr::make_xgeom(p.L, p.M, sms, device_info().smem_optin, out, sbytes, aligned);
}

// The streaming schedule (opt-in with MNB_GEMV_SCHED=stream) takes every
// shape with at least one K-unit per warp.
static bool stream_ok(const MatmulParams& p, gstr::SGeom* out) {
    const char* sc = sched_env();
    if (!sc || std::strcmp(sc, "stream") != 0) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    return gstr::make_sgeom(p.L, p.M, p.M <= 8 ? 8 : 16, sms, device_info().smem_optin, out);
}

// The persistent schedule (gemv_pers.cuh) takes the shapes it was built for:
// a row tile's K in one pass of 16 warps, enough row tiles to fill every SM at
// least twice, block boundaries on warp slices.  Measured on GB300: for
// M = 1 the per-tile grid is faster (10.5 vs 12.3 us on the int4 4096 x 11008
// decode), for M = 8 the persistent one (16.0 vs 21.6 us on the int2
// 4096 x 14336 batch), so it is the default for M >= 2.  MNB_GEMV_PERS=0 / 1
// forces either schedule.
static bool pers_ok(const MatmulParams& p, gpers::PGeom* out, int* grid) {
    const char* sc = sched_env();
    if (sc && std::strcmp(sc, "pers") == 0) {
        // forced below like MNB_GEMV_PERS=1
    } else if (sc) {
        return false;
    }
    const char* env = (sc && std::strcmp(sc, "pers") == 0) ? "1" : std::getenv("MNB_GEMV_PERS");
    if (env && env[0] == '0') return false;
    if (!(env && env[0] == '1') && p.M < 2) return false;
    const Layout& L = p.L;
    if (L.KTILES > gpers::kWarps * gpers::kMaxTPW) return false;
    const int spb = L.bs / 16;
    if (spb != 1 && spb != 2 && spb != 4 && spb != 8) return false;
    gpers::PGeom g = gpers::make_pgeom(L, p.M, p.M <= 8 ? 8 : 16);
    // raw scales / zero points by bulk copy: 16-byte rows and bases
    const int sbytes = p.scale_dtype == kF32 ? 4 : 2;
    if ((L.KB * sbytes) % 16 != 0 || (reinterpret_cast<uintptr_t>(p.scales) & 15) != 0) return false;
    if (p.zp && (L.zp_row % 16 != 0 || (reinterpret_cast<uintptr_t>(p.zp) & 15) != 0)) return false;
    g.raw_row = (size_t)L.KB * sbytes;
    g.raw_zoff = 16 * g.raw_row;
    g.raw_slot = round16(g.raw_zoff + (p.zp ? 16 * (size_t)L.zp_row : 0));
    g.total_bytes += gpers::kDepth * g.raw_slot;
    if ((g.tpw * (16 / L.bits)) % spb != 0) return false;
    if (16 * g.runs > 2 * gpers::kThreads) return false;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    if (L.NT < 2 * (int64_t)sms) return false;
    if (g.total_bytes > device_info().smem_optin) return false;
    *out = g;
    *grid = sms;
    return true;
}

static gmma::Geom geom_for(const MatmulParams& p) {
    return gmma::make_geom(p.L, p.M, p.M <= 8 ? 8 : 16);
}

bool gemv_mma_supported(const MatmulParams& p) {
    if (p.M < 1 || p.M > 16 || p.g_idx != nullptr) return false;
    if (p.act_dtype != kBF16 && p.act_dtype != kF16) return false;
    const gmma::Geom g = geom_for(p);
    // K-splits must start on quantisation-block boundaries
    if (g.C > 1 && ((int64_t)g.tiles_cta * p.L.KT) % p.L.bs != 0) return false;
    return g.total_bytes <= device_info().smem_optin && p.L.NT * g.C <= 0x7FFFFFFF;
}

cudaError_t launch_gemv_mma(const MatmulParams& p, cudaStream_t s) {
    gks::KGeom kg;
    if (ks_ok(p, &kg)) {
        switch (p.L.bits) {
            case 2: return launch_gemv_ks_b2(p, kg, s);
            case 4: return launch_gemv_ks_b4(p, kg, s);
            case 8: return launch_gemv_ks_b8(p, kg, s);
            default: return cudaErrorInvalidValue;
        }
    }
    gxr::XGeom xg;
    if (xr_ok(p, &xg)) {
        switch (p.L.bits) {
            case 2: return launch_gemv_xr_b2(p, xg, s);
            case 4: return launch_gemv_xr_b4(p, xg, s);
            case 8: return launch_gemv_xr_b8(p, xg, s);
            default: return cudaErrorInvalidValue;
        }
    }
    gstr::SGeom sg;
    if (stream_ok(p, &sg)) {
        switch (p.L.bits) {
            case 2: return launch_gemv_stream_b2(p, sg, s);
            case 4: return launch_gemv_stream_b4(p, sg, s);
            case 8: return launch_gemv_stream_b8(p, sg, s);
            default: return cudaErrorInvalidValue;
        }
    }
    gpers::PGeom pg;
    int grid = 0;
    if (pers_ok(p, &pg, &grid)) {
        switch (p.L.bits) {
            case 2: return launch_gemv_pers_b2(p, pg, grid, s);
            case 4: return launch_gemv_pers_b4(p, pg, grid, s);
            case 8: return launch_gemv_pers_b8(p, pg, grid, s);
            default: return cudaErrorInvalidValue;
        }
    }
    const gmma::Geom geo = geom_for(p);
    if (geo.total_bytes > device_info().smem_optin) return cudaErrorNotSupported;
    switch (p.L.bits) {
        case 2: return launch_gemv_mma_b2(p, geo, s);
        case 4: return launch_gemv_mma_b4(p, geo, s);
        case 8: return launch_gemv_mma_b8(p, geo, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mnb
