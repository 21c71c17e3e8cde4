// Product kernels for the format set fp4.
#include "qg_inst.cuh"
QG_DEFINE_TSET(fp4, qg::TS_FP4)
