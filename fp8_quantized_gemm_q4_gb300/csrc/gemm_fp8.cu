// gemm_fp8.cu -- placeholder translation unit for the FP8 GEMM.
#include "kernels.h"
