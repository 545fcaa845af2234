"""GB300-native sparse decode with a host-resident MLA latent cache.

The CUDA library (C ABI, ``include/ess.h``) is loaded lazily by
``host_latent_cache_gb300.ess``; importing this package alone does not
need a GPU.
"""
