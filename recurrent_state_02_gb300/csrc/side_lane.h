// A second stream and four events per host thread and device, for work that
// runs beside a call's main chain (the backward's state passes, the token walk of
// packed batches).  One set per host thread, so that calls from several threads
// never share them and a stream capture on one thread never takes in another's
// work.  Made on the first call on a device, which must not be inside a stream
// capture; nullptr if they cannot be made (the caller then runs everything on its
// own stream).
#pragma once

#include <cuda_runtime.h>

#include "kernels.h"

namespace la {

struct SideLane {
    cudaStream_t stream = nullptr;
    cudaEvent_t ev[4] = {};
    bool failed = false;
};

inline SideLane *side_lane()
{
    thread_local SideLane lanes[kMaxDevices];
    const int dev = current_device_index();
    if (dev < 0) return nullptr;
    SideLane &l = lanes[dev];
    if (!l.stream && !l.failed) {
        const cudaError_t pending = cudaPeekAtLastError();   // not ours to clear
        bool ok = cudaStreamCreateWithFlags(&l.stream, cudaStreamNonBlocking) == cudaSuccess;
        for (int i = 0; ok && i < 4; ++i) ok = cudaEventCreateWithFlags(&l.ev[i], cudaEventDisableTiming) == cudaSuccess;
        if (!ok) {
            for (cudaEvent_t &ev : l.ev)
                if (ev) cudaEventDestroy(ev), ev = nullptr;
            if (l.stream) cudaStreamDestroy(l.stream);
            l.stream = nullptr;
            l.failed = true;
            if (pending == cudaSuccess) cudaGetLastError();   // clear the error of the failed creation only
        }
    }
    return l.stream ? &l : nullptr;
}

}  // namespace la
