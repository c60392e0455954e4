// Instantiations of the conv kernel with run-time MMA loops (shapes without an
// unrolled specialisation) and the upsamplers' instantiations, whose phase
// and sub-pixel tap code stays out of the plain kernels' register budget.
#include "conv3d_tcgen05.cuh"

namespace wanvae {
namespace conv {

ConvKernelFn conv_kernel_p1_n1(int kk, int nsub);
ConvKernelFn conv_kernel_p1_n2(int kk, int nsub);
ConvKernelFn conv_kernel_p2_n1(int kk, int nsub);
ConvKernelFn conv_kernel_p2_n2(int kk, int nsub);

ConvKernelFn conv_kernel_plain(int pair, int kk, int nsub, int np) {
    ConvKernelFn fn = nullptr;
    if (pair == 2)
        fn = np == 1 ? conv_kernel_p2_n1(kk, nsub) : np == 2 ? conv_kernel_p2_n2(kk, nsub) : nullptr;
    else
        fn = np == 1 ? conv_kernel_p1_n1(kk, nsub) : np == 2 ? conv_kernel_p1_n2(kk, nsub) : nullptr;
    if (fn) return fn;
    return pair == 2 ? conv3d_tcgen05_kernel<2, 0, 0, 0, false>
                     : conv3d_tcgen05_kernel<1, 0, 0, 0, false>;
}

ConvKernelFn conv_kernel_up(int pair, int kk, int nsub, int np) {
    if (kk == 4 && nsub == 1 && np == 1)
        return pair == 2 ? conv3d_tcgen05_kernel<2, 4, 1, 1, true>
                         : conv3d_tcgen05_kernel<1, 4, 1, 1, true>;
    if (kk == 4 && nsub == 1 && np == 2)  // the temporal upsampler at 384 channels
        return pair == 2 ? conv3d_tcgen05_kernel<2, 4, 1, 2, true>
                         : conv3d_tcgen05_kernel<1, 4, 1, 2, true>;
    return pair == 2 ? conv3d_tcgen05_kernel<2, 0, 0, 0, true>
                     : conv3d_tcgen05_kernel<1, 0, 0, 0, true>;
}

}  // namespace conv
}  // namespace wanvae
