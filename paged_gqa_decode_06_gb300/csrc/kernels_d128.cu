#define HEAD_DIM 128
#include "kernels_dim.inc"
