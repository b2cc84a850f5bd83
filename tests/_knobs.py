"""DG_* tuning variables for a block of calls.  The library reads them once,
at its first call, so a change only takes effect after dg_reload_env();
this context manager sets them, reloads, and restores both on exit."""
from __future__ import annotations

import contextlib
import os

import fp16_tensor_core_gb300 as dg


@contextlib.contextmanager
def knobs(**values):
    old = {k: os.environ.get(k) for k in values}
    for k, v in values.items():
        if v is None:
            os.environ.pop(k, None)
        else:
            os.environ[k] = str(v)
    dg.dg_reload_env()
    try:
        yield
    finally:
        for k, v in old.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
        dg.dg_reload_env()
