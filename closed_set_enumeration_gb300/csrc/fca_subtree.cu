// Object-list tier of libfca (sm_103a): launches without work sharing, and the choice of slices
// and of work sharing per launch. The device code is in fca_subtree.cuh.
#include "fca_subtree.cuh"

namespace fca {

template <int NW, bool COUNT, int RW>
static int launch_subtree_nw(const SubtreeArgs &a, int sm_count, void *stream)
{
    int wpb = 0, per_sm = 0;
    size_t smem = 0;
    int e = subtree_shape<NW, COUNT, RW, false>(a.d, &wpb, &smem, &per_sm);
    if (e != (int)cudaSuccess) return e;
    // split roots into slices when there are too few roots to keep every resident warp busy
    SubtreeArgs b = a;
    const unsigned long long resident = (unsigned long long)sm_count * per_sm * wpb;
    const unsigned long long want = 4 * resident;
    const unsigned long long qn = std::max<unsigned long long>(1, a.q_count);
    b.slices = (int)std::min<unsigned long long>(MAX_SLICES, std::max<unsigned long long>(1, (want + qn - 1) / qn));
    // work sharing pays when the launch has few items per warp (its tail is then a large part of
    // it); with many short items the hand-overs cost more than they save. The counting pass runs
    // without it.
    b.share = !COUNT && a.share && a.q_count * (unsigned long long)b.slices <= 8 * resident ? 1 : 0;
    if (b.share) return launch_subtree_shared(b, NW, RW, sm_count, stream);
    return launch_subtree_kernel<NW, COUNT, RW, false>(b, sm_count, stream);
}

int launch_subtree(const SubtreeArgs &a, int nw, int sm_count, void *stream)
{
    // register-resident search width by M: R <= M relevant attributes, so M <= 64 never needs more
    // than two words per lane (a kernel without the wider paths keeps more registers free)
    const int rw = reg_words_for(a.d.m);
#define FCA_SUBTREE(NWV, CNT)                                                                   \
    (rw == 2   ? launch_subtree_nw<NWV, CNT, 2>(a, sm_count, stream)                            \
     : rw == 4 ? launch_subtree_nw<NWV, CNT, 4>(a, sm_count, stream)                            \
               : launch_subtree_nw<NWV, CNT, 8>(a, sm_count, stream))
    if (a.count_work) return nw == 1 ? FCA_SUBTREE(1, true) : FCA_SUBTREE(2, true);
    return nw == 1 ? FCA_SUBTREE(1, false) : FCA_SUBTREE(2, false);
#undef FCA_SUBTREE
}

}  // namespace fca
