// device_scope.h - run a launch on the device that owns its stream.
//
// The library links its own static CUDA runtime.  That runtime follows the
// context the caller made current (torch.cuda.set_device or cudaSetDevice in
// another runtime make the device's primary context current on the thread),
// so "the current device" is the caller's.  A stream, though, belongs to one
// device, and a launch on a stream of another device than the current one
// fails.  Each entry point therefore asks the stream for its device, and, when
// that is not the current device, makes it current for the launch (device
// attributes and occupancy are then looked up for that device too) and makes
// the caller's device current again afterwards, whether the launch succeeded
// or not.  The legacy and per-thread default streams belong to the current
// device; so does a stream under graph capture, which may not be queried
// (the runtime adapter in api.cu takes these cases without asking the stream).
//
// Header-only and templated over the runtime calls so that the host logic can
// be tested on a machine without a GPU against a fake runtime.
#pragma once

namespace tfk {

// Rt provides, each returning an error code whose value-initialised state
// (0, cudaSuccess) means success:
//   stream_device(Stream, int* device), current_device(int* device), set_device(int device).
// Fn is the launch, returning the same error type.  The first error wins: a
// launch error is reported even if restoring the device then fails too.
template <class Rt, class Stream, class Fn>
auto on_stream_device(Rt& rt, Stream stream, Fn&& launch) -> decltype(launch()) {
    using Err = decltype(launch());
    int want = 0, cur = 0;
    Err e = rt.stream_device(stream, &want);
    if (e != Err{}) return e;
    if ((e = rt.current_device(&cur)) != Err{}) return e;
    if (want == cur) return launch();
    if ((e = rt.set_device(want)) != Err{}) return e;
    const Err r = launch();
    const Err back = rt.set_device(cur);
    return r != Err{} ? r : back;
}

}  // namespace tfk
