// Instantiations of the conv kernel for CTA grouping 1 and 2 N piece(s).
#define WANVAE_PAIR 1
#define WANVAE_NP 2
#include "conv3d_kernels.inc"
