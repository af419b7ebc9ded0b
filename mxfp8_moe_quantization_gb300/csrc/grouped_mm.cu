#include "common.cuh"
#include "gemm.h"
#include "launch.h"
namespace fp8moe {
cudaError_t launch_grouped_mm(const GemmArgs& g, cudaStream_t st) { return cudaErrorNotSupported; }
}
