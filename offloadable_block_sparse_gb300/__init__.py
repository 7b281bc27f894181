"""NOSA decode-step hot path on GB300: C-ABI library libnosa.so plus its ctypes binding."""
from . import nosa  # noqa: F401
