#include "kernels.h"
namespace treeattn {
cudaError_t launch_bwd_bf16(const AttnBwdArgs&) { return cudaErrorNotSupported; }
}
