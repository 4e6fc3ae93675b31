// prefill.cu -- schedule (b): long causal prefills on tcgen05 tensor cores.
#include "internal.h"

namespace pa {

bool prefill_supported(const pa_shape& /*sh*/) { return false; }

pa_status prefill_launch(const Call& /*c*/) { return PA_ERR_UNSUPPORTED; }

}  // namespace pa
