// rope_host.cpp -- the RoPE frequency table, built on the host once (TensorSharp "Mistral 3"
// page, section 4.2 and section 7, PrecomputeConstants: the frequency table, YaRN-corrected
// when the model asks for it).  The formula and the reading of the elided ramp are stated
// with pa_rope_yarn_freqs in include/pa.h.
#include <cmath>

#include "pa.h"

extern "C" int pa_rope_yarn_freqs(float *freqs, int rope_dim, float base, float yarn_scale, int orig_ctx,
                                  float beta_fast, float beta_slow) {
    if (!freqs || rope_dim < 2 || rope_dim % 2 != 0 || !(base > 1.f) || !(yarn_scale > 0.f) || orig_ctx < 0)
        return PA_ERR_INVALID_ARG;
    const bool yarn = yarn_scale != 1.f && orig_ctx > 0;
    if (yarn && !(beta_fast > beta_slow)) return PA_ERR_INVALID_ARG;
    const double two_pi = 6.283185307179586476925286766559;
    for (int i = 0; i < rope_dim / 2; ++i) {
        double f = std::pow((double)base, -2.0 * i / rope_dim);
        if (yarn) {
            const double r = orig_ctx / (two_pi / f);  // turns over the original context
            if (r < beta_slow) {
                f = f / yarn_scale;
            } else if (r <= beta_fast) {
                const double g = (beta_fast - r) / ((double)beta_fast - beta_slow);
                f = f * (1.0 - g) + f / yarn_scale * g;
            }
        }
        freqs[i] = (float)f;
    }
    return PA_OK;
}
