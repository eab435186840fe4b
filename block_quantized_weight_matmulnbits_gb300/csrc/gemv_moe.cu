// Host side of the grouped (mixture-of-experts) GEMV (kernel in gemv_moe.cuh):
// validation, geometry and the C entry point mnb_matmul_grouped.
#include <cstdlib>
#include <cstring>

#include "gemv_ks.cuh"
#include "gemv_moe.cuh"
#include "mnb.h"

namespace mnb {

cudaError_t launch_gemv_moe_b2(const MatmulParams& p, const gmma::Geom& geo, const gmoe::MoeArgs& g,
                               unsigned groups, size_t smem_bytes, cudaStream_t s);
cudaError_t launch_gemv_moe_b4(const MatmulParams& p, const gmma::Geom& geo, const gmoe::MoeArgs& g,
                               unsigned groups, size_t smem_bytes, cudaStream_t s);
cudaError_t launch_gemv_moe_b8(const MatmulParams& p, const gmma::Geom& geo, const gmoe::MoeArgs& g,
                               unsigned groups, size_t smem_bytes, cudaStream_t s);
cudaError_t launch_gemv_ks_b2(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s, const gks::MoeKs* moe,
                              bool a8 = false);
cudaError_t launch_gemv_ks_b4(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s, const gks::MoeKs* moe,
                              bool a8 = false);
cudaError_t launch_gemv_ks_b8(const MatmulParams& p, const gks::KGeom& geo, cudaStream_t s, const gks::MoeKs* moe,
                              bool a8 = false);

}  // namespace mnb

using namespace mnb;

namespace {

// Shared memory one CTA may use so that three fit on an SM (228 KB per SM,
// 1 KB reserved per CTA).
constexpr size_t kSmemBudget = 72 * 1024;

bool valid_dt(int d) { return d == kF32 || d == kF16 || d == kBF16; }
size_t dt_bytes(int d) { return d == kF32 ? 4 : 2; }
bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

extern "C" {

mnb_status mnb_matmul_grouped(const void* x, const int32_t* ids, const void* packed_b, const void* scales,
                              const uint8_t* zero_points, void* y, int64_t T, int64_t S, int64_t E, int x_per_slot,
                              int64_t N, int64_t K, int bits, int block_size, mnb_dtype act_dtype,
                              mnb_dtype out_dtype, mnb_dtype scale_dtype, mnb_stream_t stream) {
    if (T < 0 || S < 1 || E < 1 || (x_per_slot != 0 && x_per_slot != 1)) return MNB_ERR_INVALID_ARG;
    const size_t expert_bytes = mnb_packed_size(N, K, bits, block_size);
    if (expert_bytes == 0) return MNB_ERR_INVALID_ARG;
    if (!valid_dt(act_dtype) || !valid_dt(out_dtype) || !valid_dt(scale_dtype)) return MNB_ERR_INVALID_ARG;
    if (T == 0) return MNB_OK;
    if (!x || !ids || !packed_b || !scales || !y) return MNB_ERR_INVALID_ARG;
    if (!aligned_to(x, 16) || !aligned_to(y, 16) || !aligned_to(packed_b, 256) || !aligned_to(ids, 4) ||
        !aligned_to(scales, dt_bytes(scale_dtype)))
        return MNB_ERR_INVALID_ARG;
    if (act_dtype == MNB_F32) return MNB_ERR_UNSUPPORTED;
    if (E > gmoe::kMaxExperts || T > gmoe::kMaxPairs || S > gmoe::kMaxPairs || T * S > gmoe::kMaxPairs)
        return MNB_ERR_UNSUPPORTED;  // (T and S bounded first: T * S cannot overflow)
    const int pairs = (int)(T * S);
    const int MT = pairs <= 8 ? 8 : 16;

    // Decode-sized calls (at most 8 pairs) run the K-chunk schedule, one grid row per expert
    // present (MNB_MOE_SCHED=tile keeps the per-tile kernel below)
    const char* sched = std::getenv("MNB_MOE_SCHED");
    if (pairs <= gks::kMoeMaxPairs && !(sched && std::strcmp(sched, "tile") == 0)) {
        MatmulParams q{};
        q.x = x;
        q.packed_hdr = packed_b;
        q.packed = static_cast<const uint8_t*>(packed_b) + kHeaderBytes;
        q.scales = scales;
        q.zp = zero_points;
        q.y = y;
        q.M = pairs;
        q.L.init(N, K, bits, block_size);
        q.act_dtype = act_dtype;
        q.out_dtype = out_dtype;
        q.scale_dtype = scale_dtype;
        q.bias_dtype = kF32;
        q.status = device_status_word();
        if (!q.status) return MNB_ERR_CUDA;
        gks::MoeKs mk{};
        mk.ids = ids;
        mk.pairs = pairs;
        mk.S = (int)S;
        mk.E = (int)E;
        mk.x_per_slot = x_per_slot;
        mk.expert_bytes = expert_bytes;
        mk.expert_scale_bytes = (size_t)N * (size_t)q.L.KB * dt_bytes(scale_dtype);
        mk.expert_zp_bytes = (size_t)N * (size_t)q.L.zp_row;
        const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
        gks::KGeom kg;
        bool fits = aligned_to(scales, 16) && mk.expert_scale_bytes % 16 == 0 &&
                    (!zero_points || (aligned_to(zero_points, 16) && mk.expert_zp_bytes % 16 == 0)) &&
                    gks::make_kgeom(q.L, pairs, sms, device_info().smem_optin, (int)dt_bytes(scale_dtype), &kg);
        // the active experts' row tiles end to end: at most min(pairs, E) x NT, split over the SMs
        const int64_t u_max = (pairs < E ? pairs : E) * q.L.NT;
        // (the kernel finds a row tile's expert with a float reciprocal of NT: exact for NT < 2^16)
        if (fits && q.L.NT < 65536 && u_max * (sms + 1) < (int64_t)1 << 31) {
            kg.G = (int)(u_max < sms ? u_max : sms);
            kg.max_rt = (int)((u_max + kg.G - 1) / kg.G);
            // grouped: each warp stores its whole row tiles' sums itself; the CTA's last (at most
            // kW - 1) row tiles are split over all warps, their partials in shared memory
            const int64_t rem_cap = kg.max_rt < gks::kW - 1 ? kg.max_rt : gks::kW - 1;
            kg.red_bytes = (size_t)rem_cap * gks::kW * 16 * (size_t)pairs * 4;
            kg.total_bytes = kg.x_bytes + kg.red_bytes;
            if (kg.total_bytes > device_info().smem_optin) {  // whole row tiles only
                kg.red_bytes = 0;
                kg.total_bytes = kg.x_bytes;
            }
            fits = kg.total_bytes <= device_info().smem_optin;
        } else {
            fits = false;
        }
        if (fits) {
            if (inject_launch_failure()) return MNB_ERR_CUDA;
            cudaStream_t st = (cudaStream_t)stream;
            cudaError_t e;
            switch (bits) {
                case 2: e = launch_gemv_ks_b2(q, kg, st, &mk); break;
                case 4: e = launch_gemv_ks_b4(q, kg, st, &mk); break;
                case 8: e = launch_gemv_ks_b8(q, kg, st, &mk); break;
                default: return MNB_ERR_INVALID_ARG;
            }
            if (e == cudaSuccess) return MNB_OK;
            cudaGetLastError();
            if (e != cudaErrorNotSupported) return MNB_ERR_CUDA;
            // not instantiated for this block size / scale type (nothing launched): the per-tile kernel
        }
    }

    MatmulParams p{};
    p.x = x;
    p.packed_hdr = packed_b;
    p.packed = static_cast<const uint8_t*>(packed_b) + kHeaderBytes;
    p.scales = scales;
    p.zp = zero_points;
    p.y = y;
    p.M = MT;
    p.L.init(N, K, bits, block_size);
    p.act_dtype = act_dtype;
    p.out_dtype = out_dtype;
    p.scale_dtype = scale_dtype;
    p.bias_dtype = kF32;
    p.status = device_status_word();
    if (!p.status) return MNB_ERR_CUDA;

    gmma::Geom geo = gmma::make_geom(p.L, MT, MT);
    // K-splits must start on quantisation-block boundaries (as for the plain GEMV)
    if (geo.C > 1 && ((int64_t)geo.tiles_cta * p.L.KT) % p.L.bs != 0) return MNB_ERR_UNSUPPORTED;
    if (p.L.NT * geo.C > 0x7FFFFFFF) return MNB_ERR_UNSUPPORTED;

    gmoe::MoeArgs g{};
    g.ids = ids;
    g.pairs = pairs;
    g.S = (int)S;
    g.E = (int)E;
    g.x_per_slot = x_per_slot;
    g.bitmap_words = (int)((E + 31) / 32);
    // Pairs per tile pass: the MMA's rows, fewer when the staged activation
    // rows would push a CTA past a third of the SM's shared memory.
    const size_t row_bytes = geo.xb_bytes / MT;                  // staged X of one pair row
    const size_t base_bytes = geo.total_bytes - geo.xb_bytes;    // scale entries, reduction, partials
    const size_t route_bytes = 4 * (size_t)g.bitmap_words + 4 * (size_t)pairs + 16;
    int chunk = MT < pairs ? MT : pairs;
    while (chunk > 1 && base_bytes + (size_t)chunk * row_bytes + route_bytes > kSmemBudget) --chunk;
    g.chunk = chunk;
    geo.xb_bytes = (size_t)chunk * row_bytes;
    geo.total_bytes = base_bytes + geo.xb_bytes;
    g.extra_off = round16(geo.total_bytes);
    g.expert_bytes = expert_bytes;
    g.expert_scale_bytes = (size_t)N * (size_t)p.L.KB * dt_bytes(scale_dtype);
    g.expert_zp_bytes = (size_t)N * (size_t)p.L.zp_row;
    const size_t smem = round16(g.extra_off + 4 * (size_t)g.bitmap_words + 4 * (size_t)pairs);
    if (smem > device_info().smem_optin) return MNB_ERR_UNSUPPORTED;
    // Expert sets per row tile (grid y): enough CTAs for about two waves at
    // three resident CTAs per SM, never more sets than experts that can be active.
    const int64_t max_sets = E < pairs ? E : pairs;
    const int64_t ctas = p.L.NT * geo.C;
    const int sms = device_info().sm_count > 0 ? device_info().sm_count : 148;
    int64_t sets = (2 * 3 * (int64_t)sms + ctas - 1) / ctas;
    const char* env = std::getenv("MNB_MOE_SETS");  // override (tuning)
    if (env && std::atoi(env) > 0) sets = std::atoi(env);
    if (sets > max_sets) sets = max_sets;
    if (sets < 1) sets = 1;
    const unsigned groups = (unsigned)sets;

    if (inject_launch_failure()) return MNB_ERR_CUDA;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e;
    switch (bits) {
        case 2: e = launch_gemv_moe_b2(p, geo, g, groups, smem, s); break;
        case 4: e = launch_gemv_moe_b4(p, geo, g, groups, smem, s); break;
        case 8: e = launch_gemv_moe_b8(p, geo, g, groups, smem, s); break;
        default: return MNB_ERR_INVALID_ARG;
    }
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MNB_ERR_CUDA;
    }
    return MNB_OK;
}

}  // extern "C"
