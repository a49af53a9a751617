// Single translation unit of libmoe: every kernel file is included here so
// that the device error word and other file-scope device symbols need no
// relocatable device code.
#include "route.cu"
#include "router.cu"
#include "permute.cu"
#include "plan_static.cu"
#include "quant.cu"
#include "mxfp4.cu"
#include "gemm.cu"
#include "layer.cu"
#include "gemm_mx.cu"
#include "diag.cu"
