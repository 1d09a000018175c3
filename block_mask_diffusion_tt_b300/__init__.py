"""B300-native denoiser step of the TwoTower block mask-diffusion decoder.

The compute path lives in ``libtt.so`` (hand-written CUDA for sm_103a, C ABI in
``include/tt.h``); ``block_mask_diffusion_tt_b300.tt`` is its thin ctypes
binding.  ``synth`` holds the seeded input generators.  Importing the package
loads nothing; the binding loads the library on first use and raises if it is
missing.
"""
__all__ = ["synth", "tt"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
