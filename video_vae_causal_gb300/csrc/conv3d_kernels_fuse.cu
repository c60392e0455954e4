// Instantiations of the conv kernel with the block's input norm fused into
// its halo loads: the halo plans whose one channel chunk holds all c_in
// channels (16, 32, 48, 64, 96 or 128), one N piece; run-time loops otherwise.
#include "conv3d_tcgen05.cuh"

namespace wanvae {
namespace conv {

template <int kPair>
ConvKernelFn fuse_kernel(int kk, int nsub, int np) {
#define WANVAE_FUSE_SPEC(KK_, NS_) \
    if (kk == KK_ && nsub == NS_ && np == 1) \
        return conv3d_tcgen05_kernel<kPair, KK_, NS_, 1, false, true>;
    WANVAE_FUSE_SPEC(2, 3)  // 96 channels: three 32-channel sub-tiles
    WANVAE_FUSE_SPEC(4, 1)  // 64
    WANVAE_FUSE_SPEC(4, 2)  // 128
    WANVAE_FUSE_SPEC(2, 1)  // 32
    WANVAE_FUSE_SPEC(1, 1)  // 16
    WANVAE_FUSE_SPEC(1, 3)  // 48
#undef WANVAE_FUSE_SPEC
    return conv3d_tcgen05_kernel<kPair, 0, 0, 0, false, true>;
}

ConvKernelFn conv_kernel_fuse(int pair, int kk, int nsub, int np) {
    return pair == 2 ? fuse_kernel<2>(kk, nsub, np) : fuse_kernel<1>(kk, nsub, np);
}

}  // namespace conv
}  // namespace wanvae
