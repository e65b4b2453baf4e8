"""FP64 CPU oracle for the GDN-2 prefill forward (test infrastructure only)."""
from .oracle import build, gdn2_forward, load_library, compile_c  # noqa: F401
