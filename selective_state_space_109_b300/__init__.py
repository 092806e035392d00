"""B300-native selective scan (S6): forward scan and decode state update.

The compute lives in ``libssmscan.so`` (hand-written CUDA for sm_103a behind a
C ABI declared in ``include/ssm_scan.h``).  ``selective_state_space_109_b300.ssm``
is the thin Python binding over that ABI; importing it loads the library and
raises if it is missing -- there is no CPU fallback.

``selective_state_space_109_b300.inputs`` draws the seeded synthetic inputs.
"""

__all__ = ["ssm", "inputs"]


def __getattr__(name):
    if name in ("ssm", "inputs"):
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
