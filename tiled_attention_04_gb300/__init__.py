"""GB300-native FlashAttention-2 (forward + backward) behind a C ABI.

Submodules are imported on demand so that the input generator and the build
script need neither torch nor the compiled library:

* ``binding``  -- ctypes binding of libfa.so (fa_fwd, fa_bwd, ...)
* ``autograd`` -- ``FlashAttention`` torch.autograd.Function
* ``inputs``   -- seeded synthetic inputs for the tests and the bench
* ``build``    -- nvcc build of libfa.so for sm_103a
"""
