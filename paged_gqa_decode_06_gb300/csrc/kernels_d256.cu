#define HEAD_DIM 256
#include "kernels_dim.inc"
