// libqlora.cu -- single translation unit of the library (the device error word and the
// kernels that set it must live in one device module without relocatable device code).
#include "quant.cu"
#include "gemm.cu"
#include "gemm_small.cu"
#include "gemv.cu"
#include "dropout.cu"
#include "merge.cu"
#include "api.cu"
#include "cat.cu"
#include "noalloc.cu"
#include "optim.cu"
