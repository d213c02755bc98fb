// Bookkeeping of a ring of staging buffers filled in order, shared by the kernel that
// uses it and by a host-side unit test.  Plain C++: no CUDA types.
#pragma once

#if defined(__CUDACC__)
#define PA_HOST_DEVICE __host__ __device__
#else
#define PA_HOST_DEVICE
#endif

namespace pa {

// Tile t of a stream goes to stage t % stages; it is that stage's fill number
// t / stages, and an mbarrier per stage completes one phase per fill, so fill u
// completes the phase of parity u & 1.
struct StageFill {
    bool any;         // the stage was filled at least once
    unsigned parity;  // phase parity that the stage's last fill completes
};

// The last fill of stage `st` after the first `issued` tiles were issued.  A producer
// that stops early waits on this phase of every stage before its block exits, so that
// no bulk copy is still landing in shared memory when the block's resources are
// released.
PA_HOST_DEVICE inline StageFill last_fill(int issued, int stages, int st) {
    StageFill f{false, 0u};
    if (stages <= 0 || st < 0 || st >= stages || issued <= st) return f;
    f.any = true;
    f.parity = (unsigned)(((issued - 1 - st) / stages) & 1);
    return f;
}

}  // namespace pa
