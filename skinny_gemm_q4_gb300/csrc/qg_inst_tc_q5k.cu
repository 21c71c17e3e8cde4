#define QG_TC_TYPE T_Q5K
#define QG_TC_NAME launch_tc_q5k
#include "qg_inst_tc.cuh"
