"""Which build of the library the GPU tests load: None for the default
libmtprs.so, or a path given with pytest's --mtp-library option (the
MTP_DEBUG build in tests/test_zz_gpu_debug.py).  Kept apart from gpu_util
so that CPU-only test sessions never import torch through it."""
LIBRARY = None
