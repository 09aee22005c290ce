// tmap.cuh -- the driver's tensor-map encoder (cuTensorMapEncodeTiled), looked
// up once through the runtime so the library needs no link against libcuda.
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>

namespace medusa {
// nullptr when the driver does not provide it
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
}  // namespace medusa
