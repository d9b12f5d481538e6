#include "kernels.h"
namespace treeattn {
cudaError_t launch_fwd_bf16(const AttnArgs&) { return cudaErrorNotSupported; }
}
