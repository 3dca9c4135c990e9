// placeholder: replaced by the tensor-core backward kernels
#include <cuda_runtime.h>
#include <string>
#include "internal.h"
namespace mesh {
int launch_tile_bwd_tc(const BwdArgs&, void*, std::string* err) {
  *err = "bf16 backward not built yet";
  return (int)cudaErrorNotSupported;
}
}  // namespace mesh
