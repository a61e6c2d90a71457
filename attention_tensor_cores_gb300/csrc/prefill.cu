// Row-tile attention (placeholder until the kernel lands).
#include "internal.h"
namespace fmha {
size_t prefill_workspace_bytes(const AttnArgs&) { return 0; }
int launch_prefill(const AttnArgs&, void*, size_t, cudaStream_t)
{
    return set_error(FMHA_ERR_UNSUPPORTED, "row-tile path (more than 16 query rows per key/value head) not built yet");
}
}  // namespace fmha
