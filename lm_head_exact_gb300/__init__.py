"""GB300-native fused LM-head exact sampler (FlashSampling hot path, sm_103a).

The compute lives in ``libflashsample.so`` (CUDA kernels behind a C ABI);
this package is a thin ctypes binding over it plus the seeded synthetic-input
generator.  Importing the package does not load the library; the first call
of a sampling function does, and raises if the library was not built -- there
is no CPU fallback.
"""

__all__ = ["sample", "sample_ex", "sample_chunked", "sample_unfused", "sample_host",
           "FlashSampleError", "library"]


def __getattr__(name):
    if name in __all__:
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
