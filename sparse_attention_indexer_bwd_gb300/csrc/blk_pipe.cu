// The gemm kernel with the pipeline depths the library runs: two K-tile
// stages, four tile-record slots.
#define IBWD_PIPE_KST 2
#define IBWD_PIPE_MST 4
#define IBWD_PIPE_PRIMARY 1
#include "blk_pipe.cuh"
