// Product kernels for the format set q4k_q6k (mixed QKV triple).
#include "qg_inst.cuh"
QG_DEFINE_TSET(q4k_q6k, (qg::TS_Q4K | qg::TS_Q6K))
