// Adaptive draft length: the serving-side controller of the D-sweep.
//
// SGLang's controller keeps an exponential moving average (EMA) of the
// accept length over verification rounds and switches among a few fixed
// draft lengths (1, 3 and 7 by default), each with a CUDA graph captured in
// advance, so that a switch costs next to nothing (LLM inference handbook,
// "Adaptive speculative decoding").  The pages leave the switching
// rule open; the reading taken here: the next round uses the smallest tier
// whose draft length is at least the EMA of the accept length AL =
// n_accepted + 1 (a tier D can show AL up to D + 1, so a saturated tier
// moves up and an idle one moves down), and the largest tier otherwise.
// Host code only: the controller runs between rounds on the host, which
// has to pick the graph to launch anyway.
#include <math.h>
#include <stdint.h>

#include "../../include/spec_verify.h"

extern "C" {

spec_status_t spec_adaptive_init(spec_adaptive_t *s, const int32_t *tiers, int n_tiers, float beta)
{
    if (!s || !tiers || n_tiers < 1 || n_tiers > SPEC_ADAPTIVE_MAX_TIERS || !(beta >= 0.0f) ||
        !(beta < 1.0f))
        return SPEC_ERR_INVALID_ARG;
    for (int t = 0; t < n_tiers; ++t) {
        if (tiers[t] < 0 || tiers[t] > 63) return SPEC_ERR_UNSUPPORTED;
        if (t > 0 && tiers[t] <= tiers[t - 1]) return SPEC_ERR_INVALID_ARG;   // strictly increasing
        s->tiers[t] = tiers[t];
    }
    s->n_tiers = n_tiers;
    s->beta = beta;
    s->ema = 0.0f;
    s->rounds = 0;
    s->current = n_tiers - 1;   // start at the largest tier until acceptance is seen
    return SPEC_OK;
}

int spec_adaptive_draft_len(const spec_adaptive_t *s)
{
    return s ? s->tiers[s->current] : -1;
}

int spec_adaptive_update(spec_adaptive_t *s, const int32_t *n_accepted, int B)
{
    if (!s || B < 0 || (B > 0 && !n_accepted)) return -1;
    if (B > 0) {
        double sum = 0.0;
        for (int b = 0; b < B; ++b) sum += static_cast<double>(n_accepted[b]) + 1.0;   // AL
        const float mean_al = static_cast<float>(sum / B);
        s->ema = s->rounds == 0 ? mean_al : s->beta * s->ema + (1.0f - s->beta) * mean_al;
        ++s->rounds;
    }
    int pick = s->n_tiers - 1;
    for (int t = 0; t < s->n_tiers; ++t) {
        if (static_cast<float>(s->tiers[t]) >= s->ema) {
            pick = t;
            break;
        }
    }
    s->current = pick;
    return s->tiers[pick];
}

}  // extern "C"
