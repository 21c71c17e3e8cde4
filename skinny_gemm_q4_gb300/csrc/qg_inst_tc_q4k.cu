#define QG_TC_TYPE T_Q4K
#define QG_TC_NAME launch_tc_q4k
#define QG_TC_CAPACITY
#include "qg_inst_tc.cuh"
