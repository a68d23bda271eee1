// FP8 prefill attention on tcgen05 tensor cores (kernel added separately).
#include "common.cuh"
#include "kernels.h"
