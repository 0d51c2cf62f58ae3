#define HEAD_DIM 64
#include "kernels_dim.inc"
