// Product kernels for the format set q5k.
#include "qg_inst.cuh"
QG_DEFINE_TSET(q5k, qg::TS_Q5K)
