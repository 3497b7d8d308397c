// velocity_cache.cpp - host-side schedule of the conservative DiT velocity
// cache ("perf(minimax-h3): add conservative DiT velocity reuse", TeleFuser
// PR #38, section 3): inside [start_ratio, end_ratio) of the denoising
// progress a step may skip the DiT call and reuse the previous velocity, at
// most min(max_consecutive_reuse, refresh_interval - 1) times in a row after
// each DiT call; outside the window, and before any velocity exists, the DiT
// always runs.  Host code only: the GPU side of a hit is simply the absence
// of the DiT launch.
#include <cmath>
#include <cstdint>
#include <cstdio>

#include "../../include/tfk.h"
#include "status.h"

extern "C" tfk_status tfk_velocity_cache_schedule(int32_t num_steps, double start_ratio, double end_ratio,
                                                  int32_t refresh_interval, int32_t max_consecutive_reuse,
                                                  uint8_t* reuse, int32_t* num_reuse) {
    static const char* op = "tfk_velocity_cache_schedule";
    using tfk::fail;
    if (num_steps < 0)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: num_steps = %d < 0", op, num_steps);
    if (refresh_interval < 1)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: refresh_interval = %d < 1", op, refresh_interval);
    if (max_consecutive_reuse < 0)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: max_consecutive_reuse = %d < 0", op, max_consecutive_reuse);
    if (!std::isfinite(start_ratio) || !std::isfinite(end_ratio))
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: start_ratio and end_ratio must be finite", op);
    if (start_ratio < 0.0 || end_ratio > 1.0 || start_ratio > end_ratio)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: need 0 <= start_ratio (%g) <= end_ratio (%g) <= 1", op,
                    start_ratio, end_ratio);
    if (num_steps > 0 && reuse == nullptr)
        return fail(TFK_ERR_INVALID_ARGUMENT, "%s: reuse is NULL with num_steps = %d", op, num_steps);
    const int32_t limit = max_consecutive_reuse < refresh_interval - 1 ? max_consecutive_reuse : refresh_interval - 1;
    int32_t since_dit = -1;  // reuses since the last DiT call; -1 before the first call
    int32_t hits = 0;
    for (int32_t i = 0; i < num_steps; ++i) {
        const double progress = (double)i / (double)num_steps;
        const bool window = progress >= start_ratio && progress < end_ratio;
        if (window && since_dit >= 0 && since_dit < limit) {
            reuse[i] = 1;
            ++since_dit;
            ++hits;
        } else {
            reuse[i] = 0;
            since_dit = 0;
        }
    }
    if (num_reuse) *num_reuse = hits;
    return TFK_OK;
}
