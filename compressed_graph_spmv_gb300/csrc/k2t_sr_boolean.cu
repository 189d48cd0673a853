// k2t_sr_boolean.cu -- kernel instantiations for one semiring (compiled in
// parallel with the other semirings).
#include "k2t_kernels.cuh"

namespace k2t {

LaunchFn pick_boolean(uint32_t engine, int dir, int vw)
{
    return dir == K2T_RIGHT ? pick_vw<1, K2T_RIGHT>(engine, vw) : pick_vw<1, K2T_LEFT>(engine, vw);
}

}  // namespace k2t
