// Product kernels for the format set q6k.
#include "qg_inst.cuh"
QG_DEFINE_TSET(q6k, qg::TS_Q6K)
