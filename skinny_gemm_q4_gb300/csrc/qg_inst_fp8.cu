// Product kernels for the format set fp8 (block-scaled e4m3).
#include "qg_inst.cuh"
QG_DEFINE_TSET(fp8, qg::TS_FP8)
