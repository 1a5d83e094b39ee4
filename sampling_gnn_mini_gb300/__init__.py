"""GB300 mini-batch pipeline of sampling-based GNN training.

The product is the C-ABI library ``libsg.so`` (hand-written CUDA for
sm_103a, declared in ``include/sg.h``); ``binding`` is its ctypes binding and
``pipeline`` orders the calls of one mini-batch.
"""
from . import binding  # noqa: F401
from .binding import SgError  # noqa: F401

__all__ = ["binding", "SgError"]
