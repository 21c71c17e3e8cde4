#define QG_TC_TYPE T_Q6K
#define QG_TC_NAME launch_tc_q6k
#include "qg_inst_tc.cuh"
