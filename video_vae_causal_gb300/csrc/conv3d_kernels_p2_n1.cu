// Instantiations of the conv kernel for CTA grouping 2 and 1 N piece(s).
#define WANVAE_PAIR 2
#define WANVAE_NP 1
#include "conv3d_kernels.inc"
