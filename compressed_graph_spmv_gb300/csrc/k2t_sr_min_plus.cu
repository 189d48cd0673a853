// k2t_sr_min_plus.cu -- kernel instantiations for one semiring (compiled in
// parallel with the other semirings).
#include "k2t_kernels.cuh"

namespace k2t {

LaunchFn pick_min_plus(uint32_t engine, int dir, int vw)
{
    return dir == K2T_RIGHT ? pick_vw<2, K2T_RIGHT>(engine, vw) : pick_vw<2, K2T_LEFT>(engine, vw);
}

}  // namespace k2t
