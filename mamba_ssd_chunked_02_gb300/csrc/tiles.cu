// tiles.cu -- per-shape launch choices (the "next" item of per-shape tile
// selection): a static table written by an offline sweep, consulted by the
// stage-2 and stage-4 launchers before they fall back to their launch-time
// models, and a process-global override that the sweep uses to time each
// candidate.
//
// Pages: "NVIDIA、cuTileでMamba-2フォワードパスを高速化" (ai.newsbites.today),
// the optimisation table (an autotuner picks the configuration per input);
// "NVIDIA CUDA Tile로 Mamba-2 순방향 전달 커널 가속화" (devin.kr), "cuTile 기반 성능
// 최적화 기법" (exhaustive search over block size and occupancy per input shape);
// "Accelerating Mamba-2 with High-Performance Forward Pass Kernels in NVIDIA
// CUDA Tile" (brifing.si), section 10.  The pages search at run time; here the
// search runs once, offline, and its result is compiled in.
#include <atomic>

#include "internal.h"
#include "mamba2_ssd.h"

namespace m2 {
namespace {

const TileChoice kTable[] = {
#include "tile_table.inc"
    {0, 0, 0, 0, 0, 0, 0, 0, 0, 0}   // end marker
};

std::atomic<int32_t> g_override[4] = {{0}, {0}, {0}, {0}};

constexpr int kMaxDevices = 64;
std::atomic<int> g_sms[kMaxDevices] = {};

}  // namespace

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();   // no device: nothing will launch, keep the error out of later checks
        return kFallbackSMs;
    }
    int v = g_sms[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) {
            cudaGetLastError();
            return kFallbackSMs;
        }
        g_sms[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

const TileChoice* find_tile(const Dims& d) {
    const int64_t hpg = d.G > 0 ? d.H / d.G : 0, bnc = d.b * d.nc;
    for (const TileChoice& t : kTable) {
        if (t.N == 0) break;
        if (t.N == d.N && t.P == d.P && t.L == d.L && t.hpg == hpg && bnc >= t.bnc_lo && bnc <= t.bnc_hi)
            return &t;
    }
    return nullptr;
}

int tile_override(int k) { return (k >= 0 && k < 4) ? g_override[k].load(std::memory_order_relaxed) : 0; }

}  // namespace m2

extern "C" {

mamba2_status mamba2_ssd_tile_override(int32_t stage2_units, int32_t stage4_v1, int32_t stage4_v2,
                                       int32_t stage4_waves1) {
    if (stage2_units < m2::kEvenSplit || stage4_v1 < -1 || stage4_v2 < 0 || stage4_waves1 < 0)
        return MAMBA2_ERR_INVALID_ARG;
    if (stage4_v1 <= 0 && (stage4_v2 != 0 || stage4_waves1 != 0)) return MAMBA2_ERR_INVALID_ARG;
    m2::g_override[0].store(stage2_units);
    m2::g_override[1].store(stage4_v1);
    m2::g_override[2].store(stage4_v2);
    m2::g_override[3].store(stage4_waves1);
    return MAMBA2_OK;
}

}  // extern "C"
