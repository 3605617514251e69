// The gemm kernel with the shallowest pipeline: one K-tile stage, two
// tile-record slots.  Only the test of the pipeline's ordering runs it; its
// results must be bitwise those of the production depths.
#define IBWD_PIPE_KST 1
#define IBWD_PIPE_MST 2
#define IBWD_PIPE_PRIMARY 0
#include "blk_pipe.cuh"
