// Product kernels for the format set q4k.
#include "qg_inst.cuh"
QG_DEFINE_TSET(q4k, qg::TS_Q4K)
