// sdv_depth.cu - adaptive draft depth, a host-side state machine run once per verify cycle
// ("Inside OpenJet Engine", section "Cheap drafting, careful state management": a configured
// depth is cut by one for the cycle after a rejection; "How Kinetic is fast", section "Where the
// guesses come from": draft length follows how recent drafts did, and outright misses pause
// drafting for longer and longer).  No device code: the caller feeds it the accepted count it
// already copies back for the host.
#include "sdverify.h"

namespace {

int32_t cut_depth(const sd_depth_state *s) { return s->k_max > 1 ? s->k_max - 1 : 1; }

}  // namespace

extern "C" {

sd_status sd_depth_init(sd_depth_state *s, int32_t k_max, int32_t max_pause) {
    if (!s || k_max < 1 || k_max > 15 || max_pause < 0) return SD_EINVAL;
    s->k_max = k_max;
    s->max_pause = max_pause;
    s->k_next = k_max;
    s->pause_left = 0;
    s->misses = 0;
    return SD_OK;
}

sd_status sd_depth_update(sd_depth_state *s, int32_t accepted) {
    if (!s || s->k_max < 1 || s->k_max > 15 || s->max_pause < 0) return SD_EINVAL;
    const int32_t k = s->k_next;
    if (k == 0) {  // a cycle without drafts: count the pause down
        if (s->pause_left > 0) --s->pause_left;
        s->k_next = s->pause_left > 0 ? 0 : cut_depth(s);
        return SD_OK;
    }
    if (accepted < 0 || accepted > k) return SD_EINVAL;
    if (accepted == k) {
        s->misses = 0;
        s->k_next = s->k_max;
    } else if (accepted > 0) {
        s->misses = 0;
        s->k_next = cut_depth(s);
    } else {
        if (s->misses < 31) ++s->misses;
        const int64_t len = int64_t(1) << (s->misses - 1);
        s->pause_left = static_cast<int32_t>(len < s->max_pause ? len : s->max_pause);
        s->k_next = s->pause_left > 0 ? 0 : cut_depth(s);
    }
    return SD_OK;
}

}  // extern "C"
