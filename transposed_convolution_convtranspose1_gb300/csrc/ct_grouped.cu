// ct_grouped.cu -- grouped/depthwise stride-phase gather on CUDA cores.
#include "ct_routes.h"

namespace ct {

bool grouped_supports(const Problem&) { return false; }
bool grouped_preferred(const Problem&) { return false; }
cudaError_t launch_grouped(const Problem&, const void*, const void*, const void*, void*,
                           cudaStream_t, Profile*) {
    return cudaErrorNotSupported;
}

}  // namespace ct
