#define QG_TC_TYPE T_Q4K
#define QG_TC_NAME launch_tc_q4k_q6k
#define QG_TC_MIXED
#include "qg_inst_tc.cuh"
