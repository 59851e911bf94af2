// Object-list tier of libfca (sm_103a): launches with work sharing inside blocks (compiled apart
// from the others so the two sets of kernels build in parallel). The device code is in
// fca_subtree.cuh.
#include "fca_subtree.cuh"

namespace fca {

int launch_subtree_shared(const SubtreeArgs &b, int nw, int rw, int sm_count, void *stream)
{
    if (nw == 1) {
        return rw == 2   ? launch_subtree_kernel<1, false, 2, true>(b, sm_count, stream)
               : rw == 4 ? launch_subtree_kernel<1, false, 4, true>(b, sm_count, stream)
                         : launch_subtree_kernel<1, false, 8, true>(b, sm_count, stream);
    }
    return rw == 2   ? launch_subtree_kernel<2, false, 2, true>(b, sm_count, stream)
           : rw == 4 ? launch_subtree_kernel<2, false, 4, true>(b, sm_count, stream)
                     : launch_subtree_kernel<2, false, 8, true>(b, sm_count, stream);
}

}  // namespace fca
